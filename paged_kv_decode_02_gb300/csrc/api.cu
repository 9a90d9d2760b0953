// api.cu -- the C ABI of libpagedkv.so: argument checks, launch planning, TMA
// descriptors and kernel launches. Declared (with semantics) in include/pagedkv.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "pagedkv.h"

namespace pkv {

std::atomic<unsigned long long> g_kernel_launches{0};
namespace {

constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per shared-memory copy wait
constexpr int kMaxQueryLen = PKV_MAX_QUERY_LEN;
constexpr int kTcMinRows = 48;  // multi-query rows per KV head from which tcgen05 wins
constexpr int kTcTileRows = 128;  // rows of one tcgen05 MMA (M): a KV head's row tile
// at most this many rows per KV head: two softmax threads per row (each lane quarter holds
// 16 rows twice), so that the exponentials of a tile spread over all four SM sub-partitions
constexpr int kTcSplitRows = 64;
// tcgen05 kernel: the cost of ending a KV head (its partly filled last tile, the
// epilogue, the next head's first scores) in tiles; ranges are balanced on tiles plus
// this much per head. A sweep of whole calls on GB300 (48 and 128 query rows per KV
// head, with the softmax row sums on the tensor cores) put the best at 2 (1: 8-15 %
// slower, 3: 1-3 %, 4 and 5: 3-5 %)
constexpr int kTcHeadCost = 2;
// cascade decode: the prefix kernel runs on about 1/kCascadePrefixShare of the SMs
constexpr int kCascadePrefixShare = 3;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map over a cache viewed as [num_blocks*Hkv*block_size rows, D elements]; one
// box is block_size rows by one 128-byte (64-byte for 64-byte rows) swizzle span.
bool make_cache_map(CUtensorMap* map, const void* base, bool int8, int D, long long rows,
                    int BS) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const int elt = int8 ? 1 : 2;
  const int row_bytes = D * elt;
  const int seg = row_bytes >= 128 ? 128 : 64;
  cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
  cuuint32_t box[2] = {cuuint32_t(seg / elt), cuuint32_t(BS)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(map, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          seg == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Encoded descriptors of recently used caches (the descriptor only depends on the
// base address and the shape, so a decode loop over the same cache re-uses it).
struct MapKey {
  const void* base;
  long long rows;
  int D, BS, q8;
  bool operator==(const MapKey& o) const {
    return base == o.base && rows == o.rows && D == o.D && BS == o.BS && q8 == o.q8;
  }
};
constexpr int kMapCache = 16;
std::mutex g_map_mu;
MapKey g_map_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_count = 0, g_map_next = 0;

bool cache_map(CUtensorMap* map, const void* base, bool q8, int D, long long rows, int BS) {
  const MapKey key{base, rows, D, BS, q8 ? 1 : 0};
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (int i = 0; i < g_map_count; ++i)
    if (g_map_keys[i] == key) {
      *map = g_maps[i];
      return true;
    }
  if (!make_cache_map(map, base, q8, D, rows, BS)) return false;
  g_map_keys[g_map_next] = key;
  g_maps[g_map_next] = *map;
  g_map_next = (g_map_next + 1) % kMapCache;
  if (g_map_count < kMapCache) ++g_map_count;
  return true;
}

// ---------------------------------------------------------------------------
// Launch plan
// ---------------------------------------------------------------------------
struct Plan {
  DecodeKernelInfo k;
  int g, gs, nsg, HU;
  int grid, W;
  size_t smem;
  size_t off_prefix, off_ctr, off_ml, off_o, ws_bytes;
};

pkv_status check_dims(const pkv_dims* d) {
  if (!d) return PKV_ERR_NULL;
  if (d->num_seqs < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 ||
      d->block_size <= 0 || d->num_blocks <= 0 || d->max_blocks_per_seq <= 0)
    return PKV_ERR_SHAPE;
  if (d->num_q_heads % d->num_kv_heads != 0) return PKV_ERR_SHAPE;
  if (d->head_dim != 64 && d->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (d->block_size != 16 && d->block_size != 32) return PKV_ERR_UNSUPPORTED;
  const long long rows = (long long)d->num_blocks * d->num_kv_heads * d->block_size;
  if (rows >= (1ll << 31)) return PKV_ERR_UNSUPPORTED;  // TMA row coordinates are int32
  if ((long long)d->max_blocks_per_seq * d->block_size >= (1ll << 31)) return PKV_ERR_SHAPE;
  return PKV_OK;
}

// Plans depend only on (dims, KV dtype, device); computing one queries occupancy and
// sets a kernel attribute, which costs tens of microseconds, so recent plans are kept.
struct PlanKey {
  pkv_dims d;
  int kvt, q_len, device, pair, sm_cap;
  bool operator==(const PlanKey& o) const {
    return std::memcmp(&d, &o.d, sizeof(d)) == 0 && kvt == o.kvt && q_len == o.q_len &&
           device == o.device && pair == o.pair && sm_cap == o.sm_cap;
  }
};
constexpr int kPlanCache = 16;
std::mutex g_plan_mu;
PlanKey g_plan_keys[kPlanCache];
Plan g_plans[kPlanCache];
int g_plan_count = 0, g_plan_next = 0;

pkv_status make_plan_uncached(const pkv_dims* d, int kvt, int q_len, bool pair, int sm_cap,
                              Plan* pl);

// q_len > 1: the causal multi-query decode (bf16 caches). pair: 16-token blocks go in
// pairs on the tensor-core paths (pairs start after a skipped prefix). sm_cap > 0: size
// the grid for that many SMs (the rest run another kernel at the same time).
pkv_status make_plan(const pkv_dims* d, int kvt, Plan* pl, int q_len = 1, bool pair = true,
                     int sm_cap = 0) {
  pkv_status st = check_dims(d);
  if (st != PKV_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  PlanKey key;
  std::memset(&key, 0, sizeof(key));
  key.d = *d;
  key.kvt = kvt;
  key.q_len = q_len;
  key.device = dev;
  key.pair = pair ? 1 : 0;
  key.sm_cap = sm_cap;
  std::lock_guard<std::mutex> lock(g_plan_mu);
  for (int i = 0; i < g_plan_count; ++i)
    if (g_plan_keys[i] == key) {
      *pl = g_plans[i];
      return PKV_OK;
    }
  st = make_plan_uncached(d, kvt, q_len, pair, sm_cap, pl);
  if (st != PKV_OK) return st;
  g_plan_keys[g_plan_next] = key;
  g_plans[g_plan_next] = *pl;
  g_plan_next = (g_plan_next + 1) % kPlanCache;
  if (g_plan_count < kPlanCache) ++g_plan_count;
  return PKV_OK;
}

pkv_status make_plan_uncached(const pkv_dims* d, int kvt, int q_len, bool pair, int sm_cap,
                              Plan* pl) {
  Plan P{};
  P.g = d->num_q_heads / d->num_kv_heads;
  // query rows per KV head: (new token, group member) pairs, split into work units of
  // at most 16 rows (the MMA's M) on the tensor-core path
  const int rows = q_len * P.g;
  const bool mma = P.g >= 4 || q_len > 1;
  if (mma) {
    int nsg = 1;
    while (rows % nsg != 0 || rows / nsg > 16) ++nsg;
    P.nsg = nsg;
    P.gs = rows / nsg;
  } else {
    P.nsg = 1;
    P.gs = P.g;
  }
  P.HU = d->num_kv_heads * P.nsg;
  const int simt = mma ? 0 : P.g;
  bool found = false;
  if (q_len > 1) {
    if (kvt < PKV_KV_BF16 || kvt > PKV_KV_FP8_E5M2) return PKV_ERR_DTYPE;
    // KV heads with 48 or more query rows go through the tcgen05 kernel, fewer rows
    // through the mma.sync path: measured on GB300 with the spec-70b lengths, tcgen05 vs
    // mma.sync per call: 16 rows 136.6 vs 93.4 us, 48 rows 146.4 vs 150.8, 64 rows 49.8
    // vs 72.8, 128 rows 152.4 vs 490.6 (an M = 128 MMA wastes what a small head leaves
    // empty). A head's rows are cut into nsg equal row tiles of at most 128 (the last one
    // padded when they do not divide), one tcgen05 work unit each. One-byte caches take
    // the tcgen05 kernel for every row count (it widens the codes to bf16 in shared
    // memory; the mma.sync multi-query path reads bf16 caches only).
    if ((rows >= kTcMinRows || kvt != PKV_KV_BF16) &&
        select_decode_tc(d->head_dim, d->block_size, rows > kTcTileRows, rows <= kTcSplitRows,
                         kvt, &P.k)) {
      P.nsg = (rows + kTcTileRows - 1) / kTcTileRows;
      P.gs = (rows + P.nsg - 1) / P.nsg;
      P.HU = d->num_kv_heads * P.nsg;
      found = true;
    } else if (kvt == PKV_KV_BF16) {
      found = select_decode_bf16_multi(d->head_dim, d->block_size, P.nsg, &P.k);
    }
  } else {
    switch (kvt) {
      case PKV_KV_BF16:
        found = select_decode_bf16(d->head_dim, d->block_size, simt, &P.k, pair);
        break;
      case PKV_KV_INT8:
        found = select_decode_int8(d->head_dim, d->block_size, simt, &P.k, pair);
        break;
      case PKV_KV_FP8_E4M3:
        found = select_decode_e4m3(d->head_dim, d->block_size, simt, &P.k, pair);
        break;
      case PKV_KV_FP8_E5M2:
        found = select_decode_e5m2(d->head_dim, d->block_size, simt, &P.k, pair);
        break;
      default: return PKV_ERR_DTYPE;
    }
  }
  if (!found) return PKV_ERR_UNSUPPORTED;
  // shared-memory rings per CTA: one per warp, or one per worker of nsg warps; the
  // tcgen05 kernel: its fixed layout plus the tile prefix and lengths of the batch
  const int rings = P.k.coop ? P.k.warps / P.nsg : P.k.warps;
  P.smem = P.k.tc ? size_t(P.k.warp_smem) + size_t(12) * (d->num_seqs + 1)
                  : size_t(rings) * P.k.warp_smem + 1024 +
                        align_up(size_t(d->num_seqs + 1) * 4, 16);

  int dev = 0, sms = 0, per_sm = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, P.k.fn) != cudaSuccess) return PKV_ERR_CUDA;
  // tcgen05 kernel: every CTA's range start, [grid + 1] (grid <= SMs)
  if (P.k.tc) P.smem += size_t(8) * (sms + 1);
  const size_t max_dyn = size_t(optin) - fa.sharedSizeBytes;
  if (P.smem > max_dyn) return PKV_ERR_UNSUPPORTED;  // batch too large for one CTA's table
  // the attribute is an upper bound only: set it to the most any batch size may need,
  // so that cached plans of other batch sizes stay launchable
  if (cudaFuncSetAttribute(P.k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(max_dyn)) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, P.k.fn, P.k.warps * 32, P.smem) !=
          cudaSuccess ||
      per_sm <= 0)
    return PKV_ERR_CUDA;
  if (P.k.tc) per_sm = 1;  // 512 TMEM columns per CTA: one CTA per SM
  P.grid = (sm_cap > 0 ? std::min(sm_cap, sms) : sms) * per_sm;
  // owners of partial slots: decode warps (warps left idle by a cooperative CTA own
  // none), or the CTAs of the tcgen05 kernel
  P.W = P.k.tc ? P.grid : (P.k.coop ? P.grid * rings * P.nsg : P.grid * P.k.warps);

  // workspace: [prefix (B+1) int32][partial (m, l) 2W*gs float2][partial o 2W*gs*D float]
  P.off_prefix = 0;  // [B+1] work prefix, then [B+1] weighted prefix (tcgen05 kernel)
  // [B, HU] counters of the in-kernel stream-K fixups (single-token decode: one per KV
  // head; the tcgen05 kernel: one per unit)
  P.off_ctr = align_up(size_t(d->num_seqs + 1) * 8, 256);
  P.off_ml = align_up(P.off_ctr + size_t(d->num_seqs) * P.HU * 8, 256);
  P.off_o = align_up(P.off_ml + size_t(2) * P.W * P.gs * 8, 256);
  P.ws_bytes = align_up(P.off_o + size_t(2) * P.W * P.gs * d->head_dim * 4, 256);
  *pl = P;
  return PKV_OK;
}

// counters (optional): where the in-kernel fixup keeps its [B, Hkv] counter words,
// counter_words of them, instead of its region of the workspace.
pkv_status run_decode(int kvt, void* out, const void* q, const void* k_cache,
                      const void* v_cache, const float* k_scale, const float* v_scale,
                      const int32_t* block_tables, const int32_t* context_lens, float scale,
                      const pkv_dims* d, void* workspace, size_t workspace_bytes,
                      int32_t* status, cudaStream_t stream, int q_len = 1,
                      unsigned long long* counters = nullptr, size_t counter_words = 0) {
  pkv_status st = check_dims(d);
  if (st != PKV_OK) return st;
  if (q_len < 1 || q_len > kMaxQueryLen) return PKV_ERR_SHAPE;
  if (d->num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PKV_ERR_NULL;
  const bool q8 = kvt != PKV_KV_BF16;
  if (q8 && (!k_scale || !v_scale)) return PKV_ERR_NULL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (q8 && (!aligned16(k_scale) || !aligned16(v_scale))))
    return PKV_ERR_ALIGNMENT;
  Plan P;
  st = make_plan(d, kvt, &P, q_len);
  if (st != PKV_OK) return st;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < P.ws_bytes)
    return PKV_ERR_WORKSPACE;
  if (counters && ((reinterpret_cast<uintptr_t>(counters) & 7u) != 0 ||
                   size_t(d->num_seqs) * d->num_kv_heads > counter_words))
    return PKV_ERR_WORKSPACE;

  const long long rows = (long long)d->num_blocks * d->num_kv_heads * d->block_size;
  CUtensorMap tmk, tmv;
  if (!cache_map(&tmk, k_cache, q8, d->head_dim, rows, d->block_size) ||
      !cache_map(&tmv, v_cache, q8, d->head_dim, rows, d->block_size))
    return PKV_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams p{};
  p.q = q;
  p.out = out;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.part_o = reinterpret_cast<float*>(ws + P.off_o);
  p.part_ml = reinterpret_cast<float*>(ws + P.off_ml);
  p.prefix_out = reinterpret_cast<int32_t*>(ws + P.off_prefix);
  p.fix_ctr = counters ? counters : reinterpret_cast<unsigned long long*>(ws + P.off_ctr);
  // single-token decode without a status word folds its cut units in the decode
  // kernel (the last warp to finish a unit); otherwise the merge kernel does
  // (the tcgen05 kernel: every call without a status word whose fold weights, one per
  // part and row with at most one part per CTA, fit its six idle tile buffers)
  const bool tc_fold = P.k.tc && P.grid <= 1024 && size_t(8192) + size_t(4) * P.grid * P.gs <=
                                     size_t(6) * (d->head_dim / 64) * 128 * 128;
  p.fixup = ((P.k.fixup && q_len == 1 && P.nsg == 1) || tc_fold) && status == nullptr ? 1 : 0;
  p.status = status;
  p.B = d->num_seqs;
  p.Hq = d->num_q_heads;
  p.Hkv = d->num_kv_heads;
  p.MBS = d->max_blocks_per_seq;
  p.NB = d->num_blocks;
  p.g = P.g;
  p.gs = P.gs;
  p.nsg = P.nsg;
  p.HU = P.HU;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = kTimeoutNs;
  p.skip = 0;
  p.unit_slot0 = -1;
  p.q_len = q_len;
  p.beta = P.k.tc ? kTcHeadCost : 0;

  // tcgen05 kernel: whole units leave through TMA tensor stores of g-row boxes when g is
  // 8, 16 or 32 and the row tiles start on tokens (each box then starts on a 1024-byte
  // swizzle atom of the staged rows)
  CUtensorMap tmo;
  std::memset(&tmo, 0, sizeof(tmo));
  // (a split tile stages 16 rows per lane quarter: g up to 16)
  if (P.k.tc && (P.g == 8 || P.g == 16 || (P.g == 32 && P.gs > kTcSplitRows)) &&
      P.gs % P.g == 0 &&
      cache_map(&tmo, out, false, d->head_dim,
                (long long)d->num_seqs * q_len * d->num_q_heads, P.g))
    p.tma_out = 1;
  void* args3[] = {&tmk, &tmv, &p};
  void* args4[] = {&tmk, &tmv, &tmo, &p};
  if (launch_pdl(P.k.fn, dim3(P.grid), dim3(P.k.warps * 32), P.k.tc ? args4 : args3, P.smem,
                 stream) != cudaSuccess)
    return PKV_ERR_CUDA;

  MergeParams m{};
  m.out = out;
  m.part_o = p.part_o;
  m.part_ml = p.part_ml;
  m.prefix = p.prefix_out;
  m.block_tables = block_tables;
  m.context_lens = context_lens;
  m.status = status;
  m.MBS = p.MBS;
  m.NB = p.NB;
  m.BS = d->block_size;
  m.B = p.B;
  m.Hq = p.Hq;
  m.D = d->head_dim;
  m.q_len = q_len;
  m.g = P.g;
  m.gs = P.gs;
  m.nsg = P.nsg;
  m.HU = P.HU;
  m.W = P.k.tc ? P.W : P.W / P.nsg;  // CTAs, or workers of nsg warps
  m.beta = p.beta;
  m.wprefix = p.prefix_out + (d->num_seqs + 1);
  if (!p.fixup) launch_merge(m, stream);  // else cut units were folded in the kernel
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}

// ---------------------------------------------------------------------------
// Cascade (shared prefix) decode
// ---------------------------------------------------------------------------
struct CascadePlan {
  Plan dec;                    // suffix decode (its partial arrays get 2W + B*HU slots)
  int R, nsplit, per_split, overlap;
  PrefixKernelInfo pk;
  size_t off_prefix, off_ml, off_o, off_pre_o, off_pre_ml, ws_bytes;
};

pkv_status make_cascade_plan(const pkv_dims* d, int prefix_blocks, CascadePlan* cp,
                             int kvt = PKV_KV_BF16) {
  pkv_status st = check_dims(d);
  if (st != PKV_OK) return st;
  if (kvt < PKV_KV_BF16 || kvt > PKV_KV_FP8_E5M2) return PKV_ERR_DTYPE;
  if (prefix_blocks < 1 || prefix_blocks > d->max_blocks_per_seq) return PKV_ERR_SHAPE;
  if (!select_prefix_kernel(d->head_dim, d->block_size, kvt, &cp->pk))
    return PKV_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  cp->R = d->num_seqs * (d->num_q_heads / d->num_kv_heads);
  // One prefix CTA per SM (TMEM and shared memory), grid (row tile, KV head, split),
  // cut at tile boundaries. The prefix kernel and the suffix decode are independent:
  // the prefix takes about a third of the SMs (at least one CTA per row tile and KV
  // head, at most half) and the suffix decode, sized for the other SMs, runs beside it.
  // When the row tiles alone need more than half the SMs, the two run one after the
  // other and the prefix splits to fill one wave.
  const int ctas = ((cp->R + cp->pk.rows - 1) / cp->pk.rows) * d->num_kv_heads;
  const int tiles = (prefix_blocks + cp->pk.tile_blocks - 1) / cp->pk.tile_blocks;
  const int max_tiles = cp->pk.max_split_blocks / cp->pk.tile_blocks;
  const int min_split = (tiles + max_tiles - 1) / max_tiles;
  cp->overlap = ctas * min_split <= sms / 2 ? 1 : 0;
  const int budget = cp->overlap ? std::max(ctas * min_split, sms / kCascadePrefixShare) : sms;
  const int nsplit =
      std::max(min_split, std::max(1, std::min(tiles, budget / std::max(1, ctas))));
  cp->per_split = ((tiles + nsplit - 1) / nsplit) * cp->pk.tile_blocks;
  cp->nsplit = (prefix_blocks + cp->per_split - 1) / cp->per_split;
  st = make_plan(d, kvt, &cp->dec, 1, true, cp->overlap ? sms - ctas * cp->nsplit : 0);
  if (st != PKV_OK) return st;
  const Plan& P = cp->dec;
  const size_t nslots = size_t(2) * P.W + size_t(d->num_seqs) * P.HU;
  cp->off_prefix = 0;
  cp->off_ml = align_up(size_t(d->num_seqs + 1) * 4, 256);
  cp->off_o = align_up(cp->off_ml + nslots * P.gs * 8, 256);
  cp->off_pre_o = align_up(cp->off_o + nslots * P.gs * d->head_dim * 4, 256);
  const size_t recs = size_t(cp->nsplit) * d->num_kv_heads * cp->R;
  cp->off_pre_ml = align_up(cp->off_pre_o + recs * d->head_dim * 4, 256);
  cp->ws_bytes = align_up(cp->off_pre_ml + recs * 8, 256);
  if (cudaFuncSetAttribute(cp->pk.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, cp->pk.smem) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

pkv_status run_cascade(int kvt, void* out, const void* q, const void* k_cache,
                       const void* v_cache, const float* k_scale, const float* v_scale,
                       const int32_t* block_tables, const int32_t* context_lens,
                       int prefix_blocks, float scale, const pkv_dims* d, void* workspace,
                       size_t workspace_bytes, int32_t* status, cudaStream_t stream) {
  pkv_status st = check_dims(d);
  if (st != PKV_OK) return st;
  if (d->num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_NULL;
  const bool q8 = kvt != PKV_KV_BF16;
  if (q8 && (!k_scale || !v_scale)) return PKV_ERR_NULL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (q8 && (!aligned16(k_scale) || !aligned16(v_scale))))
    return PKV_ERR_ALIGNMENT;
  CascadePlan C;
  st = make_cascade_plan(d, prefix_blocks, &C, kvt);
  if (st != PKV_OK) return st;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < C.ws_bytes)
    return PKV_ERR_WORKSPACE;
  const Plan& P = C.dec;
  const long long rows = (long long)d->num_blocks * d->num_kv_heads * d->block_size;
  CUtensorMap tmk, tmv;
  if (!cache_map(&tmk, k_cache, q8, d->head_dim, rows, d->block_size) ||
      !cache_map(&tmv, v_cache, q8, d->head_dim, rows, d->block_size))
    return PKV_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const float scale_log2 = scale * 1.4426950408889634f;

  // 1. the shared prefix, once per KV head for all B*g query rows
  PrefixParams pp{};
  pp.q = q;
  pp.k_scale = k_scale;
  pp.v_scale = v_scale;
  pp.prefix_ids = block_tables;  // row 0 holds the shared prefix
  pp.pre_o = reinterpret_cast<float*>(ws + C.off_pre_o);
  pp.pre_ml = reinterpret_cast<float*>(ws + C.off_pre_ml);
  pp.P = prefix_blocks;
  pp.B = d->num_seqs;
  pp.Hq = d->num_q_heads;
  pp.Hkv = d->num_kv_heads;
  pp.g = P.g;
  pp.R = C.R;
  pp.NB = d->num_blocks;
  pp.nsplit = C.nsplit;
  pp.overlap = C.overlap;
  pp.per_split = C.per_split;
  pp.scale_log2 = scale_log2;
  pp.timeout_ns = kTimeoutNs;
  pp.status = status;
  {
    void* args[] = {&tmk, &tmv, &pp};
    if (launch_pdl(C.pk.fn, dim3((C.R + C.pk.rows - 1) / C.pk.rows, d->num_kv_heads, C.nsplit),
                   dim3(C.pk.threads), args, C.pk.smem, stream) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  // 2. the private suffixes: the ordinary decode over the tables past the prefix; a
  //    complete unit leaves its partial in slot 2W + s*HU + u
  DecodeParams p{};
  p.q = q;
  p.out = out;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.part_o = reinterpret_cast<float*>(ws + C.off_o);
  p.part_ml = reinterpret_cast<float*>(ws + C.off_ml);
  p.prefix_out = reinterpret_cast<int32_t*>(ws + C.off_prefix);
  p.status = status;
  p.B = d->num_seqs;
  p.Hq = d->num_q_heads;
  p.Hkv = d->num_kv_heads;
  p.MBS = d->max_blocks_per_seq;
  p.NB = d->num_blocks;
  p.g = P.g;
  p.gs = P.gs;
  p.nsg = P.nsg;
  p.HU = P.HU;
  p.scale_log2 = scale_log2;
  p.timeout_ns = kTimeoutNs;
  p.skip = prefix_blocks;
  p.unit_slot0 = 2 * P.W;
  p.late_wait = C.overlap;
  p.q_len = 1;
  {
    void* args[] = {&tmk, &tmv, &p};
    if (launch_pdl(P.k.fn, dim3(P.grid), dim3(P.k.warps * 32), args, P.smem, stream) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
  }
  // 3. fold prefix and suffix partials
  CascadeMergeParams m{};
  m.out = out;
  m.part_o = p.part_o;
  m.part_ml = p.part_ml;
  m.pre_o = pp.pre_o;
  m.pre_ml = pp.pre_ml;
  m.prefix = p.prefix_out;
  m.block_tables = block_tables;
  m.context_lens = context_lens;
  m.status = status;
  m.B = p.B;
  m.Hq = p.Hq;
  m.Hkv = p.Hkv;
  m.D = d->head_dim;
  m.MBS = p.MBS;
  m.NB = p.NB;
  m.BS = d->block_size;
  m.P = prefix_blocks;
  m.g = P.g;
  m.gs = P.gs;
  m.nsg = P.nsg;
  m.HU = P.HU;
  m.W = P.W;
  m.Wg = P.W / P.nsg;
  m.R = C.R;
  m.nsplit = C.nsplit;
  launch_cascade_merge(m, stream);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}

pkv_status check_append(const void* k, const void* v, const void* kc, const void* vc,
                        const int64_t* slots, int T, const pkv_dims* d) {
  pkv_status st = check_dims(d);
  if (st != PKV_OK) return st;
  if (T < 0) return PKV_ERR_SHAPE;
  if (T == 0) return PKV_OK;
  if (!k || !v || !kc || !vc || !slots) return PKV_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(kc) || !aligned16(vc)) return PKV_ERR_ALIGNMENT;
  return PKV_OK;
}

}  // namespace

pkv_status decode_bf16_fixed_counters(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, float scale,
                                      const pkv_dims* dims, void* workspace,
                                      size_t workspace_bytes, unsigned long long* counters,
                                      size_t counter_words, int32_t* status,
                                      cudaStream_t stream) {
  if (!counters) return PKV_ERR_NULL;
  return run_decode(PKV_KV_BF16, out, q, k_cache, v_cache, nullptr, nullptr, block_tables,
                    context_lens, scale, dims, workspace, workspace_bytes, status, stream, 1,
                    counters, counter_words);
}

}  // namespace pkv

using namespace pkv;

namespace pkv {
namespace {

// Element sizes of a block move for a KV dtype: bytes per cache element, and whether
// there are scale arrays.
bool move_layout(int kvt, int* elt, bool* scales) {
  switch (kvt) {
    case PKV_KV_BF16: *elt = 2; *scales = false; return true;
    case PKV_KV_INT8:
    case PKV_KV_FP8_E4M3:
    case PKV_KV_FP8_E5M2: *elt = 1; *scales = true; return true;
    default: return false;
  }
}

// The device address of a pinned host buffer (the same address under unified
// addressing); false for pageable or unknown memory.
bool host_device_ptr(const void* host, void** dev) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return false;
  *dev = attr.devicePointer;
  return true;
}

enum MoveKind { kCopy, kSwapOut, kSwapIn };

// cache arrays: k, v, ks, vs (device); other: host arrays in the same order (swap) or
// unused (copy).
pkv_status run_move(MoveKind kind, void* const cache[4], void* const other[4],
                    const int32_t* src_ids, const int32_t* dst_ids, int32_t n, int kvt,
                    const pkv_dims* d, int32_t* status, cudaStream_t stream) {
  if (!d) return PKV_ERR_NULL;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 || d->block_size <= 0 ||
      d->num_blocks <= 0 || n < 0)
    return PKV_ERR_SHAPE;
  int elt = 0;
  bool scales = false;
  if (!move_layout(kvt, &elt, &scales)) return PKV_ERR_DTYPE;
  if (n == 0) return PKV_OK;
  const int narrays = scales ? 4 : 2;
  const long long rows = (long long)d->num_kv_heads * d->block_size;
  const long long chunk[4] = {rows * d->head_dim * elt, rows * d->head_dim * elt, rows * 4,
                              rows * 4};
  for (int i = 0; i < narrays; ++i) {
    if (chunk[i] % 16 != 0 || chunk[i] / 16 >= (1ll << 31)) return PKV_ERR_UNSUPPORTED;
    if (!cache[i] || (kind != kCopy && !other[i])) return PKV_ERR_NULL;
    if (!aligned16(cache[i]) || (kind != kCopy && !aligned16(other[i])))
      return PKV_ERR_ALIGNMENT;
  }
  if ((kind != kSwapIn && !src_ids) || (kind != kSwapOut && !dst_ids)) return PKV_ERR_NULL;
  MoveParams p{};
  p.narrays = narrays;
  p.n = n;
  p.NB = d->num_blocks;
  p.status = status;
  p.src_ids = kind == kSwapIn ? nullptr : src_ids;
  p.dst_ids = kind == kSwapOut ? nullptr : dst_ids;
  for (int i = 0; i < narrays; ++i) {
    void* host = nullptr;
    if (kind != kCopy && !host_device_ptr(other[i], &host)) return PKV_ERR_HOST_MEMORY;
    const void* src = kind == kSwapIn ? host : cache[i];
    void* dst = kind == kSwapOut ? host : cache[i];
    p.arrays[i].src = static_cast<const uint4*>(src);
    p.arrays[i].dst = static_cast<uint4*>(dst);
    p.arrays[i].chunk16 = int(chunk[i] / 16);
  }
  return launch_block_move(p, stream) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace
}  // namespace pkv

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_NULL: return "PKV_ERR_NULL: a required pointer is NULL";
    case PKV_ERR_DTYPE: return "PKV_ERR_DTYPE: unknown KV dtype";
    case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE: sizes are invalid or inconsistent";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: head_dim/block_size/batch not built";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA call failed";
    case PKV_ERR_ALIGNMENT: return "PKV_ERR_ALIGNMENT: a device pointer is not 16-byte aligned";
    case PKV_ERR_HOST_MEMORY: return "PKV_ERR_HOST_MEMORY: a host buffer is not pinned host memory";
  }
  return "unknown pkv_status";
}

int pkv_version(void) { return 100; }

uint64_t pkv_kernel_launch_count(void) {
  return g_kernel_launches.load(std::memory_order_relaxed);
}

pkv_status pkv_append_bf16(const void* k, const void* v, void* k_cache, void* v_cache,
                           const int64_t* slot_mapping, int32_t num_tokens,
                           const pkv_dims* dims, pkv_stream_t stream) {
  pkv_status st = check_append(k, v, k_cache, v_cache, slot_mapping, num_tokens, dims);
  if (st != PKV_OK || num_tokens == 0) return st;
  if (launch_append_bf16(k, v, k_cache, v_cache, slot_mapping, num_tokens, dims->num_kv_heads,
                         dims->head_dim, dims->block_size, dims->num_blocks,
                         reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

pkv_status pkv_append_int8(const void* k, const void* v, int8_t* k_cache, int8_t* v_cache,
                           float* k_scale, float* v_scale, const int64_t* slot_mapping,
                           int32_t num_tokens, const pkv_dims* dims, pkv_stream_t stream) {
  pkv_status st = check_append(k, v, k_cache, v_cache, slot_mapping, num_tokens, dims);
  if (st != PKV_OK || num_tokens == 0) return st;
  if (!k_scale || !v_scale) return PKV_ERR_NULL;
  if (launch_append_q8(CODE_I8, k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, num_tokens,
                         dims->num_kv_heads, dims->head_dim, dims->block_size, dims->num_blocks,
                         reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

pkv_status pkv_decode_workspace_bytes(const pkv_dims* dims, pkv_kv_dtype kv_dtype,
                                      size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  if (kv_dtype < PKV_KV_BF16 || kv_dtype > PKV_KV_FP8_E5M2) return PKV_ERR_DTYPE;
  Plan P;
  pkv_status st = make_plan(dims, kv_dtype, &P);
  if (st != PKV_OK) return st;
  *bytes = P.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_decode_bf16(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens,
                           float scale, const pkv_dims* dims, void* workspace,
                           size_t workspace_bytes, int32_t* status, pkv_stream_t stream) {
  return run_decode(PKV_KV_BF16, out, q, k_cache, v_cache, nullptr, nullptr, block_tables,
                    context_lens, scale, dims, workspace, workspace_bytes, status,
                    reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_decode_cascade_workspace_bytes(const pkv_dims* dims, int32_t prefix_blocks,
                                              size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  CascadePlan C;
  pkv_status st = make_cascade_plan(dims, prefix_blocks, &C);
  if (st != PKV_OK) return st;
  *bytes = C.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_decode_cascade_bf16(void* out, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables,
                                   const int32_t* context_lens, int32_t prefix_blocks,
                                   float scale, const pkv_dims* dims, void* workspace,
                                   size_t workspace_bytes, int32_t* status, pkv_stream_t stream) {
  return run_cascade(PKV_KV_BF16, out, q, k_cache, v_cache, nullptr, nullptr, block_tables,
                     context_lens, prefix_blocks, scale, dims, workspace, workspace_bytes, status,
                     reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_decode_cascade_q8_workspace_bytes(const pkv_dims* dims, int32_t prefix_blocks,
                                                 pkv_kv_dtype kv_dtype, size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  if (kv_dtype != PKV_KV_INT8 && kv_dtype != PKV_KV_FP8_E4M3 && kv_dtype != PKV_KV_FP8_E5M2)
    return PKV_ERR_DTYPE;
  CascadePlan C;
  pkv_status st = make_cascade_plan(dims, prefix_blocks, &C, kv_dtype);
  if (st != PKV_OK) return st;
  *bytes = C.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_decode_cascade_q8(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const float* k_scale, const float* v_scale,
                                 const int32_t* block_tables, const int32_t* context_lens,
                                 int32_t prefix_blocks, float scale, pkv_kv_dtype kv_dtype,
                                 const pkv_dims* dims, void* workspace, size_t workspace_bytes,
                                 int32_t* status, pkv_stream_t stream) {
  if (kv_dtype != PKV_KV_INT8 && kv_dtype != PKV_KV_FP8_E4M3 && kv_dtype != PKV_KV_FP8_E5M2)
    return PKV_ERR_DTYPE;
  return run_cascade(kv_dtype, out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                     context_lens, prefix_blocks, scale, dims, workspace, workspace_bytes, status,
                     reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_decode_int8(void* out, const void* q, const int8_t* k_cache,
                           const int8_t* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* block_tables, const int32_t* context_lens,
                           float scale, const pkv_dims* dims, void* workspace,
                           size_t workspace_bytes, int32_t* status, pkv_stream_t stream) {
  return run_decode(PKV_KV_INT8, out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                    context_lens,
                    scale, dims, workspace, workspace_bytes, status,
                    reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_append_fp8(const void* k, const void* v, uint8_t* k_cache, uint8_t* v_cache,
                          float* k_scale, float* v_scale, const int64_t* slot_mapping,
                          int32_t num_tokens, pkv_kv_dtype fp8_format, const pkv_dims* dims,
                          pkv_stream_t stream) {
  if (fp8_format != PKV_KV_FP8_E4M3 && fp8_format != PKV_KV_FP8_E5M2) return PKV_ERR_DTYPE;
  pkv_status st = check_append(k, v, k_cache, v_cache, slot_mapping, num_tokens, dims);
  if (st != PKV_OK || num_tokens == 0) return st;
  if (!k_scale || !v_scale) return PKV_ERR_NULL;
  const int code = fp8_format == PKV_KV_FP8_E4M3 ? CODE_E4M3 : CODE_E5M2;
  if (launch_append_q8(code, k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, num_tokens,
                       dims->num_kv_heads, dims->head_dim, dims->block_size, dims->num_blocks,
                       reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

pkv_status pkv_decode_fp8(void* out, const void* q, const uint8_t* k_cache,
                          const uint8_t* v_cache, const float* k_scale, const float* v_scale,
                          const int32_t* block_tables, const int32_t* context_lens, float scale,
                          pkv_kv_dtype fp8_format, const pkv_dims* dims, void* workspace,
                          size_t workspace_bytes, int32_t* status, pkv_stream_t stream) {
  if (fp8_format != PKV_KV_FP8_E4M3 && fp8_format != PKV_KV_FP8_E5M2) return PKV_ERR_DTYPE;
  return run_decode(fp8_format, out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                    context_lens, scale, dims, workspace, workspace_bytes, status,
                    reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_decode_multi_workspace_bytes(const pkv_dims* dims, int32_t q_len,
                                            size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  if (q_len < 1 || q_len > kMaxQueryLen) return PKV_ERR_SHAPE;
  Plan P;
  pkv_status st = make_plan(dims, PKV_KV_BF16, &P, q_len);
  if (st != PKV_OK) return st;
  *bytes = P.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_decode_multi_bf16(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, int32_t q_len, float scale,
                                 const pkv_dims* dims, void* workspace, size_t workspace_bytes,
                                 int32_t* status, pkv_stream_t stream) {
  return run_decode(PKV_KV_BF16, out, q, k_cache, v_cache, nullptr, nullptr, block_tables,
                    context_lens, scale, dims, workspace, workspace_bytes, status,
                    reinterpret_cast<cudaStream_t>(stream), q_len);
}

pkv_status pkv_decode_multi_q8_workspace_bytes(const pkv_dims* dims, int32_t q_len,
                                               pkv_kv_dtype kv_dtype, size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  if (kv_dtype != PKV_KV_INT8 && kv_dtype != PKV_KV_FP8_E4M3 && kv_dtype != PKV_KV_FP8_E5M2)
    return PKV_ERR_DTYPE;
  if (q_len < 1 || q_len > kMaxQueryLen) return PKV_ERR_SHAPE;
  Plan P;
  pkv_status st = make_plan(dims, kv_dtype, &P, q_len);
  if (st != PKV_OK) return st;
  *bytes = P.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_decode_multi_q8(void* out, const void* q, const void* k_cache,
                               const void* v_cache, const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, const int32_t* context_lens,
                               int32_t q_len, float scale, pkv_kv_dtype kv_dtype,
                               const pkv_dims* dims, void* workspace, size_t workspace_bytes,
                               int32_t* status, pkv_stream_t stream) {
  if (kv_dtype != PKV_KV_INT8 && kv_dtype != PKV_KV_FP8_E4M3 && kv_dtype != PKV_KV_FP8_E5M2)
    return PKV_ERR_DTYPE;
  return run_decode(kv_dtype, out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                    context_lens, scale, dims, workspace, workspace_bytes, status,
                    reinterpret_cast<cudaStream_t>(stream), q_len);
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                           const int32_t* src_ids, const int32_t* dst_ids, int32_t num_pairs,
                           pkv_kv_dtype kv_dtype, const pkv_dims* dims, int32_t* status,
                           pkv_stream_t stream) {
  void* cache[4] = {k_cache, v_cache, k_scale, v_scale};
  void* none[4] = {nullptr, nullptr, nullptr, nullptr};
  return run_move(kCopy, cache, none, src_ids, dst_ids, num_pairs, kv_dtype, dims, status,
                  reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_swap_out(void* host_k, void* host_v, float* host_k_scale, float* host_v_scale,
                        const void* k_cache, const void* v_cache, const float* k_scale,
                        const float* v_scale, const int32_t* block_ids, int32_t num_blocks_moved,
                        pkv_kv_dtype kv_dtype, const pkv_dims* dims, int32_t* status,
                        pkv_stream_t stream) {
  void* cache[4] = {const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                    const_cast<float*>(k_scale), const_cast<float*>(v_scale)};
  void* host[4] = {host_k, host_v, host_k_scale, host_v_scale};
  return run_move(kSwapOut, cache, host, block_ids, nullptr, num_blocks_moved, kv_dtype, dims,
                  status, reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_swap_in(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                       const void* host_k, const void* host_v, const float* host_k_scale,
                       const float* host_v_scale, const int32_t* block_ids,
                       int32_t num_blocks_moved, pkv_kv_dtype kv_dtype, const pkv_dims* dims,
                       int32_t* status, pkv_stream_t stream) {
  void* cache[4] = {k_cache, v_cache, k_scale, v_scale};
  void* host[4] = {const_cast<void*>(host_k), const_cast<void*>(host_v),
                   const_cast<float*>(host_k_scale), const_cast<float*>(host_v_scale)};
  return run_move(kSwapIn, cache, host, nullptr, block_ids, num_blocks_moved, kv_dtype, dims,
                  status, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
