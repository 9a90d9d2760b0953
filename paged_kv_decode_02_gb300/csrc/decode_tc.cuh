// decode_tc.cuh -- paged decode attention on the fifth-generation tensor cores
// (instantiated per KV dtype in decode_tc.cu, decode_tc_int8.cu, decode_tc_e4m3.cu and
// decode_tc_e5m2.cu).
//
// What is computed is the decode attention of decode.cuh: for every sequence s, KV
// head h and query row r of that head (q_len new tokens x g query heads; new token i
// sees the first L - q_len + 1 + i cached tokens, the causal rule of speculative
// verification in "推测解码" of "大模型工程（五）：推理优化核心技法", chenk.top),
//   out[r] = softmax(scale * K q_r) V
// over the tokens reached through the block table ("分页注意力", same page).
//
// The q_len * g rows of a KV head are cut into nsg equal row tiles of gs <= 128 rows
// (one tile up to 128 rows; a chunk of chunked prefill, q_len up to 256, takes
// several), and each row tile goes through one M = 128 tcgen05 MMA per KV tile, so a
// KV block is multiplied once for every 128 rows instead of once per 16-row subgroup.
// A work unit is (KV head, row tile): unit u of a sequence is KV head u / nsg, rows
// (u % nsg) * gs .. + gs - 1. The row tiles of one head are consecutive units, so
// their re-reads of the head's blocks come from L2. Work: the flat order (sequence,
// unit, tile of 128 tokens) is cut into one contiguous range per CTA (one CTA per SM).
// Within a range the tiles of one unit form a segment; a segment covering the whole
// unit writes the output, a cut one (only a range's first and last can be) leaves an
// unnormalised (o, m, l) record per row in slot 2c (the first segment of CTA c) or
// 2c + 1 (the last). Without a status word the CTA that completes a cut unit folds its
// records at its end (tc_tail_fixup); with one, the split-KV merge kernel validates
// and folds.
// Roles per CTA (224 threads; 352 with the warps 7..10 below), as in the cascade
// prefix kernel:
//   warp 0 / warp 6: TMA copies of the K / V tiles into two-stage rings (one box per
//                    16- or 32-token block and 64-column slab, lane b copies block b;
//                    block ids are read one tile ahead);
//   warp 1:          TMEM allocation; one thread issues every MMA:
//                    S_t = Q K_t^T (fp32, two TMEM buffers), O += P_t V_t (A = P in TMEM)
//                    and l += P_t 1 (the row sums of the bf16 weights, P times a ones
//                    tile in shared memory), so the normalisation uses exactly the
//                    weights P.V used and the softmax warps add nothing up;
//   warps 2..5:      one query row per thread: Q rows of each segment into shared
//                    memory, softmax with the causal and context masks, P to TMEM,
//                    the segment's epilogue from O and l in TMEM. A unit of at most 64
//                    rows runs split (CS = 2): each lane quarter holds 16 rows twice and
//                    the two threads of a row take half of each tile's columns, so the
//                    exponentials spread over all four SM sub-partitions (measured on
//                    GB300, spec-70b with 48 rows per head: 103.2 -> 97.2 us per call).
//   warps 7..10:     bf16 caches, D = 128, more than 64 rows (PAIR): the second softmax
//                    warp of each lane quarter, the two of a quarter taking half of each
//                    row's columns and sharing its tile maximum (measured on GB300:
//                    chunk-70b 341.5 -> 321.8 us, spec-70b-q16 105.5 -> 104.2 us per
//                    call); one-byte caches: the converters below.
// The softmax keeps a reference maximum per row that moves only when a tile's maximum
// exceeds it by more than 8 (log2 units); O and l are then rescaled in TMEM before the
// next P.V. Every wait is bounded: on a timeout the CTA sets a status bit, lets its
// copies and MMAs complete, frees its TMEM and leaves.
//
// One-byte caches (INT8, FP8 E4M3 / E5M2 codes with one fp32 scale per token and KV
// head: "KV 缓存量化" of the chenk.top page): the producers land a tile's codes and
// scales in the upper part of the tile's bf16 buffer and a scale area; four converter
// warps (7..10) widen the codes exactly (Code8), multiply by the row's scale and write
// the bf16 values over the whole buffer in the layout the MMA reads, so that K and V
// enter the same bf16 MMAs dequantised (one bf16 rounding of code x scale, as a bf16
// cache holds its values). Rows past the context become zeros there.
#pragma once

#include "convert.cuh"
#include "decode.cuh"
#include "fold.cuh"
#include "tcgen05.cuh"

namespace pkv {

// 16-byte asynchronous copy global -> shared (zero fill when src_bytes is 0); the
// copies of a thread complete at cp_async_wait_all.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <int D, int BS, bool Q8 = false, bool PAIR = false>
struct TcDecode {
  static constexpr int kM = 128;               // query rows per MMA (rows of a KV head, padded)
  static constexpr int kN = 128;               // tokens per tile
  static constexpr int kBlocks = kN / BS;      // blocks per tile
  static constexpr int kSlabs = D / 64;        // 128-byte column slabs of a row
  static constexpr int kSlab = kN * 128;       // one slab of a tile (== kM * 128)
  static constexpr int kTile = kSlabs * kSlab; // a Q, K or V tile
  static constexpr int kOffQ = 0;              // Q x2 (segment parity)
  static constexpr int kOffK = kOffQ + 2 * kTile;
  static constexpr int kOffV = kOffK + 2 * kTile;
  // all-ones B operand (16 x 128 tokens, K-major) of the MMA that sums the rows of P
  static constexpr int kOffOnes = kOffV + 2 * kTile;
  // one-byte caches: a tile's codes land in the last kCodeTile bytes of its 16-bit
  // buffer; its scales in kN fp32 slots: K scales in four (tile i in slot i % 4: the
  // softmax of tile i reads them, and tile i + 4's copy only starts once it has), then V
  // scales in two (the stage's, read by the converters only)
  static constexpr int kCodeTile = kN * D;
  static constexpr int kCodeOff = kTile - kCodeTile;
  static constexpr int kScaleBytes = kN * 4;
  static constexpr int kOffScales = kOffOnes + 4096;
  // paired softmax warps (bf16 caches, so no scales): the halves of each row's tile
  // maximum, [2 tiles][2 halves][128 rows] fp32
  static constexpr int kOffXmax = kOffScales;
  static constexpr int kOffBar = kOffScales + (Q8 ? 6 * kScaleBytes : PAIR ? 2048 : 0);
  // mbarriers: kfull[2] kempty[2] vfull[2] vempty[2] sfull[2] pfull ofull mdone qfull[2] ofree
  // (+ one-byte caches: kstage[2] vstage[2], the copies of the codes; kscale[4], the K
  // scales of slot i % 4 ready for the softmax; paired softmax warps: xmax[4], both
  // halves of a lane quarter's tile maxima written)
  static constexpr int kNumBars = Q8 ? 24 : PAIR ? 20 : 16;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  // [2] cut segments of this CTA (first, last) for the tail fixup: s, h, n, tiles, state
  static constexpr int kOffCut = kOffAbort + 12;
  // [B+1] tile prefix, [B+1] weighted prefix (tiles + beta per non-empty sequence),
  // [B] clamped lengths
  static constexpr int kOffTables = kOffCut + 48;
  // + 8 * (grid + 1) + 12 * (B + 1) at run time
  static constexpr int kFixedSmem = kOffTables + 1024;
  // warps: 0 K copies, 1 MMA, 2..5 softmax, 6 V copies (+ 7..10 converters, or the
  // second softmax warp of each lane quarter)
  static constexpr int kThreads = (Q8 || PAIR) ? 352 : 224;
  static constexpr int kSoftThreads = PAIR ? 256 : 128;
  static constexpr uint32_t kTmemCols = 512;
  // S x2, O, P (bf16 pairs), l (row sums of P, fp32; 16 columns written by its MMA)
  static constexpr int kColS = 0, kColO = 2 * kN, kColP = 2 * kN + 128, kColL = kColP + kN / 2;
  static_assert(kColL + 16 <= int(kTmemCols) && kColO + D <= kColP, "TMEM columns");
  static_assert(kOffOnes % 1024 == 0, "swizzle atom alignment");
  static_assert(kN % BS == 0 && D % 64 == 0 && kSlab == kM * 128, "tile shape");
  static_assert(kOffTables % 16 == 0 && kOffCut % 16 == 0, "table alignment");
  static_assert(!(Q8 && PAIR) && (!PAIR || D == 128), "paired softmax: bf16, D = 128");
};

// Position in the flat (sequence, unit, tile) order; a unit is (KV head, row tile).
struct TileCursor {
  int s, h, j, n;  // sequence, unit, tile of the unit, tiles per unit of the sequence
};

__device__ __forceinline__ void tile_locate(TileCursor& c, long long f, const int* prefix, int B,
                                            int U) {
  int lo = 0, hi = B;  // U*prefix[lo] <= f < U*prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((long long)U * prefix[mid] <= f) lo = mid; else hi = mid;
  }
  c.s = lo;
  c.n = prefix[lo + 1] - prefix[lo];
  const long long rem = f - (long long)U * prefix[lo];
  c.h = int(rem / c.n);
  c.j = int(rem % c.n);
}

__device__ __forceinline__ void tile_next(TileCursor& c, const int* prefix, int B, int U) {
  if (++c.j < c.n) return;
  c.j = 0;
  if (++c.h < U) return;
  c.h = 0;
  do { ++c.s; } while (c.s < B && prefix[c.s + 1] == prefix[c.s]);
  c.n = c.s < B ? prefix[c.s + 1] - prefix[c.s] : 0;
}

// Tiles of the flat (sequence, unit, tile) order before weighted position x (U units
// per sequence). Ranges are equal cuts of a weighted order in which unit (s, h)
// takes tiles_s + beta positions (its tiles, then beta for the cost of ending a unit);
// a range covers the tiles whose positions fall in it. prefix / wprefix: exclusive
// prefixes of the tiles and of the weights per sequence.
__device__ __forceinline__ long long tc_tiles_before(long long x, const int* prefix,
                                                     const int* wprefix, int B, int U,
                                                     int beta) {
  if (x >= (long long)U * wprefix[B]) return (long long)U * prefix[B];
  int lo = 0, hi = B;  // U*wprefix[lo] <= x < U*wprefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((long long)U * wprefix[mid] <= x) lo = mid; else hi = mid;
  }
  const int n = prefix[lo + 1] - prefix[lo];
  const long long rem = x - (long long)U * wprefix[lo];
  const long long h = rem / (n + beta), o = rem % (n + beta);
  return (long long)U * prefix[lo] + h * n + min(o, (long long)n);
}

// Stream-K fixup at the end of a CTA (no merge kernel follows). A KV head is cut only
// where a range ends inside it, so a CTA holds at most two cut segments (its first and
// its last), whose unnormalised (o, m, l) records are in slots 2c and 2c + 1. After its
// last tile the CTA fences its records and adds the tiles of each cut segment to the
// head's counter; the CTA whose addition completes the head's n tiles folds every part
// of it with the online-softmax rescaling, all threads together: first per row the
// largest m, l = sum 2^(m_i - m) l_i and each part's weight 2^(m_i - m) / l (in the
// idle Q, K and V tile buffers: 8 KiB + 4 * parts * rows bytes), then per 16-byte
// output quad the weighted sum of the parts' o.
// The parts are the segments of the CTAs whose ranges hold the head's tiles: the first
// one's last segment (its first when its range starts at the head), then the first
// segments of the CTAs whose non-empty ranges start inside the head. A counter word
// holds a launch tag (launch_tag: a 40-bit hash of the grid's launch number) over a
// 24-bit tile count: a word with another tag counts as zero, so the workspace needs no clearing,
// and the completing CTA resets it. Writers order their records before the counter
// update (a barrier, then a fence by the counting thread), the completing thread fences
// after it and, past a barrier, every thread reads the records through L2.
template <int D, bool kTiles>
__device__ __forceinline__ void tc_tail_fixup(const DecodeParams& p, const int* s_prefix,
                                              const long long* s_rs, volatile int* cut,
                                              uint8_t* scratch, int nthreads) {
  const int tid = threadIdx.x, C = gridDim.x, R = p.gs, U = p.HU;
  if (!(cut[4] | cut[9])) return;  // no cut segment (uniform: shared memory after a barrier)
  __syncthreads();                 // every thread's records are written
  if (tid < 2 && cut[5 * tid + 4]) {
    // release: the fence of the counting thread orders the records the barrier ordered
    // before it ahead of its counter update (one thread waits, not every thread)
    __threadfence();
    volatile int* e = cut + 5 * tid;
    const int s = e[0], h = e[1], n = e[2], mine = e[3];
    const unsigned long long tag = launch_tag();
    unsigned long long* ctr = p.fix_ctr + size_t(s) * U + h;
    // first guess: every other part already counted, the usual state for the CTA that
    // completes the head (a wrong guess costs one more round, as reading it would)
    unsigned long long cur = (tag << 24) | unsigned(n - mine);
    int last = 0;
    for (;;) {
      const unsigned long long base = (cur >> 24) == tag ? (cur & 0xffffffull) : 0ull;
      const unsigned long long want = (tag << 24) | (base + unsigned(mine));
      const unsigned long long seen = atomicCAS(ctr, cur, want);
      if (seen == cur) {
        last = int(base) + mine == n;
        break;
      }
      cur = seen;
    }
    if (last) {
      __threadfence();  // acquire: the other parts' records, for every thread after the barrier
      atomicExch(ctr, 0ull);
    }
    e[4] = last ? 2 : 0;
  }
  __syncthreads();
  int* parts = reinterpret_cast<int*>(scratch);          // [C] part slots
  volatile int* s_np = parts + 1024;                      // part count
  float* wts = reinterpret_cast<float*>(scratch + 8192);  // [parts][R] weights
  constexpr int Q = D / 4;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  const float4* po = reinterpret_cast<const float4*>(p.part_o);
  __nv_bfloat16* outb = reinterpret_cast<__nv_bfloat16*>(p.out);
  for (int ei = 0; ei < 2; ++ei) {
    if (cut[5 * ei + 4] != 2) continue;
    const int s = cut[5 * ei], h = cut[5 * ei + 1], n = cut[5 * ei + 2];
    if (tid == 0) {  // the parts: slots of the CTAs whose ranges hold tiles [u0, u1)
      const long long u0 = (long long)U * s_prefix[s] + (long long)h * n, u1 = u0 + n;
      int lo = 0, hi = C;  // s_rs[lo] <= u0 < s_rs[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_rs[mid] <= u0) lo = mid; else hi = mid;
      }
      int np = 0;
      parts[np++] = 2 * lo + (s_rs[lo] < u0 ? 1 : 0);
      for (int c2 = lo + 1; c2 < C && s_rs[c2] < u1; ++c2)
        if (s_rs[c2 + 1] > s_rs[c2]) parts[np++] = 2 * c2;
      *s_np = np;
    }
    __syncthreads();
    const int np = *s_np;
    // per row: the largest m, l and every part's weight
    for (int r = tid; r < R; r += nthreads) {
      float M = -INFINITY, L = 0.f;
      for (int i0 = 0; i0 < np; i0 += 8) {
        float2 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          v[k] = i0 + k < np ? __ldcg(ml + size_t(parts[i0 + k]) * R + r)
                             : make_float2(-INFINITY, 0.f);
        float cm = v[0].x;
#pragma unroll
        for (int k = 1; k < 8; ++k) cm = fmaxf(cm, v[k].x);
        if (cm > M) {
          L *= fast_exp2(M - cm);  // 0 while nothing was folded in
          M = cm;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (i0 + k < np) wts[(i0 + k) * R + r] = v[k].x;
          if (v[k].x > -INFINITY) L = fmaf(fast_exp2(v[k].x - M), v[k].y, L);
        }
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int i = 0; i < np; ++i) {
        const float m = wts[i * R + r];
        wts[i * R + r] = m > -INFINITY ? fast_exp2(m - M) * inv : 0.f;
      }
    }
    __syncthreads();
    // per output quad: the weighted sum of the parts, 8 quads per thread at a time with
    // the loads of two parts in flight together
    const int items = R * Q;
    for (int k0 = tid; k0 < items; k0 += 8 * nthreads) {
      float4 acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i0 = 0; i0 < np; i0 += 2) {
        float4 x[8][2];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int k = k0 + j * nthreads, r = k / Q, dq = k % Q;
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2)
            x[j][c2] = (k < items && i0 + c2 < np)
                           ? __ldcg(po + (size_t(parts[i0 + c2]) * R + r) * Q + dq)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int k = k0 + j * nthreads, r = min(k / Q, R - 1);
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const float w = i0 + c2 < np ? wts[(i0 + c2) * R + r] : 0.f;
            acc[j].x = fmaf(w, x[j][c2].x, acc[j].x);
            acc[j].y = fmaf(w, x[j][c2].y, acc[j].y);
            acc[j].z = fmaf(w, x[j][c2].z, acc[j].z);
            acc[j].w = fmaf(w, x[j][c2].w, acc[j].w);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int k = k0 + j * nthreads;
        if (k >= items) break;
        const int r = k / Q, dq = k % Q;
        size_t orow;
        if constexpr (kTiles) {
          // unit h: KV head h / nsg, rows from (h % nsg) * R
          const int Rg = (h % p.nsg) * R + r;
          if (Rg >= p.q_len * p.g) continue;  // past the last row of a partial row tile
          orow = (size_t(s) * p.q_len + Rg / p.g) * p.Hq + size_t(h / p.nsg) * p.g + Rg % p.g;
        } else {
          orow = (size_t(s) * p.q_len + r / p.g) * p.Hq + size_t(h) * p.g + r % p.g;
        }
        reinterpret_cast<uint2*>(outb + orow * D)[dq] =
            make_uint2(pack_bf16x2(acc[j].x, acc[j].y), pack_bf16x2(acc[j].z, acc[j].w));
      }
    }
    __syncthreads();  // the scratch of the next entry
  }
}

// kTiles: a KV head's rows run as several row tiles (nsg > 1). The single-tile
// instantiation keeps its own index arithmetic: measured on GB300, the general form
// made the one-tile calls 17 % slower (spec-70b 102.4 -> 120.1 us) although it computes
// the same values. CODE: -1 for bf16 caches, else the one-byte code format.
template <int D, int BS, bool kTiles, int CODE = -1, int CS = 1, bool PAIR = false>
__global__ void __launch_bounds__(TcDecode<D, BS, (CODE >= 0), PAIR>::kThreads, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                           const __grid_constant__ CUtensorMap tmv,
                           const __grid_constant__ CUtensorMap tmo, const DecodeParams p) {
  constexpr bool kQ8 = CODE >= 0;
  using K = TcDecode<D, BS, kQ8, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + K::kOffAbort);
  // [grid + 1] first tile of every CTA's range, then the per-sequence tables
  long long* s_rs = reinterpret_cast<long long*>(gbase + K::kOffTables);
  int* s_prefix = reinterpret_cast<int*>(s_rs + gridDim.x + 1);
  volatile int* s_cut = reinterpret_cast<volatile int*>(gbase + K::kOffCut);
  // U units per sequence: KV head u / nsg, row tile u % nsg of gs rows (rows = q_len * g)
  const int B = p.B, Hkv = p.Hkv, beta = p.beta, U = p.HU, nsg = kTiles ? p.nsg : 1;
  const int rows = p.q_len * p.g;
  int* s_wpre = s_prefix + (B + 1);
  int* s_len = s_wpre + (B + 1);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto bar = [&](int i) { return base + K::kOffBar + 8 * i; };
  auto kfull = [&](int st) { return bar(st); };
  auto kempty = [&](int st) { return bar(2 + st); };
  auto vfull = [&](int st) { return bar(4 + st); };
  auto vempty = [&](int st) { return bar(6 + st); };
  auto sfull = [&](int st) { return bar(8 + st); };
  const uint32_t pfull = bar(10), ofull = bar(11), mdone = bar(12), ofree = bar(15);
  auto qfull = [&](int b) { return bar(13 + b); };
  // one-byte caches: the codes' copies land on kstage / vstage, and kfull / vfull
  // complete when the converters have written the bf16 values
  auto kstage = [&](int st) { return bar(16 + st); };
  auto vstage = [&](int st) { return bar(18 + st); };
  // K scales of tile i: slot i % 4; V scales of tile i: slot 4 + i % 2
  auto scale_area = [&](bool is_k, int i) {
    return base + K::kOffScales + uint32_t(is_k ? (i & 3) : 4 + (i & 1)) * K::kScaleBytes;
  };
  auto kscale = [&](int i) { return bar(20 + (i & 3)); };
  // paired softmax: both warps of lane quarter q have written their tile maxima
  auto xmax = [&](int q) { return bar(16 + q); };
  const uint32_t tmem_slot = base + K::kOffTmemSlot;

  pdl_wait_prior_grid();
  if (tid == 0) {
    for (int i = 0; i < 10; ++i) mbar_init(bar(i), 1);
    mbar_init(pfull, K::kSoftThreads);
    mbar_init(ofull, 1);
    mbar_init(mdone, 1);
    mbar_init(qfull(0), K::kSoftThreads);
    mbar_init(qfull(1), K::kSoftThreads);
    mbar_init(ofree, K::kSoftThreads);
    if constexpr (kQ8)
      for (int i = 16; i < 24; ++i) mbar_init(bar(i), 1);
    if constexpr (PAIR)
      for (int q = 0; q < 4; ++q) mbar_init(xmax(q), 64);
    *abort_flag = 0;
    s_cut[4] = s_cut[9] = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, K::kTmemCols);
  for (int k = tid; k < 4096 / 16; k += K::kThreads)  // 1.0 everywhere (bf16, or fp16)
    tc::sts128(base + K::kOffOnes + 16 * k,
               kQ8 ? make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u)   // fp16 1.0
                   : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u)); // bf16
  fence_proxy_async_smem();  // for the MMAs that read it

  // ---- tiles per sequence, their exclusive prefix, the weighted prefix (tiles plus
  //      beta per non-empty sequence), clamped lengths (every CTA) ----
  {
    const int per = (B + K::kThreads - 1) / K::kThreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int sum = 0, wsum = 0;
    for (int i = b0; i < b1; ++i) {
      const int L = min(max(__ldg(p.context_lens + i), 0), p.MBS * BS);
      s_len[i] = L;
      const int n = (L + K::kN - 1) / K::kN;
      sum += n;
      wsum += n + (n > 0 ? beta : 0);
    }
    int incl = sum, wincl = wsum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      const int wy = __shfl_up_sync(0xffffffffu, wincl, off);
      if (lane >= off) {
        incl += y;
        wincl += wy;
      }
    }
    __shared__ int warp_tot[K::kThreads / 32], warp_wtot[K::kThreads / 32];
    if (lane == 31) {
      warp_tot[warp] = incl;
      warp_wtot[warp] = wincl;
    }
    __syncthreads();
    int run = incl - sum, wrun = wincl - wsum;
    for (int w2 = 0; w2 < warp; ++w2) {
      run += warp_tot[w2];
      wrun += warp_wtot[w2];
    }
    for (int i = b0; i < b1; ++i) {
      const int n = (s_len[i] + K::kN - 1) / K::kN;
      run += n;
      wrun += n + (n > 0 ? beta : 0);
      s_prefix[i + 1] = run;
      s_wpre[i + 1] = wrun;
    }
    if (tid == 0) s_prefix[0] = s_wpre[0] = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (blockIdx.x == 0)
    for (int i = tid; i <= B; i += K::kThreads) {
      p.prefix_out[i] = s_prefix[i];
      p.prefix_out[B + 1 + i] = s_wpre[i];
    }
  if (p.fixup)  // no merge kernel follows: sequences without a tile get zeros here
    for (int s2 = blockIdx.x; s2 < B; s2 += gridDim.x) {
      if (s_prefix[s2 + 1] != s_prefix[s2]) continue;
      const int chunks = p.q_len * p.Hq * (D / 8);
      uint4* o = reinterpret_cast<uint4*>(p.out) + size_t(s2) * chunks;
      for (int k = tid; k < chunks; k += K::kThreads) o[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + K::kOffTmemSlot);

  // This CTA's tiles. Ranges are equal cuts of the weighted order, in which KV head
  // (s, h) takes tiles_s + beta positions (its tiles, then beta for the cost of ending
  // a head); a range covers the tiles whose positions fall in it. Tiles before
  // weighted position x:
  // every CTA's range start (equal cuts of the weighted order), all threads at once
  const long long TW = (long long)U * s_wpre[B];
  const int C = gridDim.x, c = blockIdx.x;
  for (int c2 = tid; c2 <= C; c2 += K::kThreads)
    s_rs[c2] = tc_tiles_before(TW * c2 / C, s_prefix, s_wpre, B, U, beta);
  __syncthreads();
  const long long ra = s_rs[c], rb = s_rs[c + 1];
  const int cnt = int(rb - ra);
  const int R = p.gs;  // query rows per unit (a row tile of the KV head's q_len * g rows)

  if (cnt > 0 && (warp == 0 || warp == 6)) {
    // ---------------- TMA producers: warp 0 streams K, warp 6 streams V ----------------
    const bool is_k = warp == 0;
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    const uint32_t region = base + (is_k ? K::kOffK : K::kOffV);
    const int rows_total = p.NB * Hkv * BS;  // a box at this row is all zero fill
    TileCursor cur;
    tile_locate(cur, ra, s_prefix, B, U);
    // lane b: physical block of block b of the tile at the cursor (rows_total: none)
    auto block_row = [&](const TileCursor& t) -> int {
      const int blk = t.j * K::kBlocks + lane;
      if (lane >= K::kBlocks || t.s >= B || blk * BS >= s_len[t.s]) return rows_total;
      int phys = __ldg(p.block_tables + size_t(t.s) * p.MBS + blk);
      phys = (phys < 0 || phys >= p.NB) ? 0 : phys;  // never copy outside the pool
      return (phys * Hkv + (kTiles ? t.h / nsg : t.h)) * BS;
    };
    int row = block_row(cur);
    int issued = 0;
    // the barrier a tile's copies complete on: the tile itself (bf16), or the staged
    // codes and scales the converters wait for (one-byte caches)
    auto copy_bar = [&](int st) {
      return kQ8 ? (is_k ? kstage(st) : vstage(st)) : (is_k ? kfull(st) : vfull(st));
    };
    for (int i = 0; i < cnt; ++i) {
      const int st = i & 1;
      const uint32_t fb = copy_bar(st);
      if (i >= 2 &&
          !__all_sync(0xffffffffu, tc::wait_or_abort(is_k ? kempty(st) : vempty(st),
                                                     uint32_t((i >> 1) - 1) & 1u, p.timeout_ns,
                                                     abort_flag)))
        break;
      if constexpr (kQ8) {
        if (lane == 0) mbar_arrive_expect_tx(fb, K::kCodeTile + K::kScaleBytes);
        __syncwarp();
        // a block past the context copies zero-filled codes and block 0's scales (its
        // rows become zeros in the conversion; the scales only have to be readable)
        const int row0 = __shfl_sync(0xffffffffu, row, 0);
        if (lane < K::kBlocks) {
          tma_load_2d(region + st * K::kTile + K::kCodeOff + lane * BS * D, map, fb, 0, row);
          const float* sc = is_k ? p.k_scale : p.v_scale;
          bulk_load(scale_area(is_k, i) + lane * BS * 4,
                    sc + size_t(row == rows_total ? row0 : row), BS * 4, fb);
        }
      } else {
        if (lane == 0) mbar_arrive_expect_tx(fb, K::kTile);
        __syncwarp();
        if (lane < K::kBlocks) {
          const uint32_t dst = region + st * K::kTile + lane * BS * 128;
#pragma unroll
          for (int sl = 0; sl < K::kSlabs; ++sl)
            tma_load_2d(dst + sl * K::kSlab, map, fb, sl * 64, row);
        }
      }
      issued = i + 1;
      tile_next(cur, s_prefix, B, U);
      if (i + 1 < cnt) row = block_row(cur);  // next tile's ids, a tile ahead
    }
    if (lane == 0)  // every copy issued must have landed before the CTA may exit
      for (int j = max(0, issued - 2); j < issued; ++j)
        mbar_wait_bounded(copy_bar(j & 1), uint32_t(j >> 1) & 1u, p.timeout_ns);
    __syncwarp();
  } else if (cnt > 0 && warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16<128, K::kN, false>();
      // P.V and the row sums run on fp16 weights and values for one-byte caches
      constexpr uint32_t kIdO =
          kQ8 ? tc::idesc_f16<128, D, true>() : tc::idesc_bf16<128, D, true>();
      constexpr uint32_t kIdL =
          kQ8 ? tc::idesc_f16<128, 16, false>() : tc::idesc_bf16<128, 16, false>();
      // Shared-memory descriptors, built once: the start address sits in the low 14 bits
      // (address >> 4, every operand below 256 KiB), so the descriptor of base + off is
      // the base's descriptor + off / 16. Measured on GB300, a thread that builds the
      // descriptors before each MMA issues one every ~125-165 cycles, while the tensor
      // cores finish an M = 128, N = 128, K = 16 step every 64 cycles.
      constexpr uint32_t kTileDesc = K::kTile >> 4;
      const uint64_t desc_q = tc::sdesc_sw128(base + K::kOffQ, 16, 1024);
      const uint64_t desc_k = tc::sdesc_sw128(base + K::kOffK, 16, 1024);
      const uint64_t desc_v = tc::sdesc_sw128(base + K::kOffV, K::kSlab, 1024);
      const uint64_t desc_ones = tc::sdesc_sw128(base + K::kOffOnes, 16, 1024);
      // S_i = Q K_i^T into score buffer i & 1 (its inputs known to be ready)
      auto mma_s = [&](int i, int qb) {
        const int st = i & 1;
        tc::fence_after_sync();
        const uint64_t qd = desc_q + qb * kTileDesc, kd = desc_k + st * kTileDesc;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          constexpr uint32_t kSlabDesc = K::kSlab >> 4;
          const uint32_t ko = (kk >> 2) * kSlabDesc + (kk & 3) * 2;  // (koff) / 16
          tc::mma_bf16(tmem + K::kColS + st * K::kN, qd + ko, kd + ko, kIdS, kk > 0 ? 1u : 0u);
        }
        tc::commit(sfull(st));
        tc::commit(kempty(st));
      };
      // P.V of tile i; the first P.V of a segment overwrites O
      auto mma_pv = [&](int i, bool seg_first) {
        const int st = i & 1;
        tc::fence_after_sync();
        const uint64_t vd = desc_v + st * kTileDesc;
#pragma unroll
        for (int kk = 0; kk < K::kN / 16; ++kk) {
          tc::mma_bf16_tmem_a(tmem + K::kColO, tmem + K::kColP + kk * 8, vd + kk * 128, kIdO,
                              (!seg_first || kk > 0) ? 1u : 0u);
          // the row sums of the bf16 weights this P.V used, next to O (same rescaling)
          tc::mma_bf16_tmem_a(tmem + K::kColL, tmem + K::kColP + kk * 8,
                              desc_ones + (kk >> 2) * 128 + (kk & 3) * 2, kIdL,
                              (!seg_first || kk > 0) ? 1u : 0u);
        }
        tc::commit(vempty(st));
        tc::commit(ofull);
      };
      // MMAs go out in the order their inputs become ready, not strictly tile by tile,
      // so that scores never wait behind a P.V whose V tile is still in flight
      // (measured on GB300: in strict order the softmax warps spent a third of their
      // time waiting for scores, most of it behind late V tiles). With pdone softmax
      // passes observed (pfull), np P.V and ns score MMAs issued:
      //   S_ns  once K_ns has landed, its score buffer is free (pass ns - 2 observed:
      //         pdone >= ns - 1) and, first in a segment, that segment's Q is ready;
      //   PV_np once pass np is observed, V_np has landed and, first in a segment, the
      //         previous segment's epilogue has read O (ofree).
      // A pass i + 1 cannot complete before PV_i, hence before pass i is observed, and
      // ns <= pdone + 1 <= np + 2, so no barrier can run two phases past the one polled.
      TileCursor sc, pc;  // tiles of the next S and the next P.V
      tile_locate(sc, ra, s_prefix, B, U);
      pc = sc;
      int ns = 0, np = 0, pdone = 0, sseg = -1, pseg = -1;
      uint32_t idle = 0;
      uint64_t t_idle = 0;
      while (np < cnt) {
        bool prog = false;
        if (pdone < ns && mbar_test_wait(pfull, uint32_t(pdone) & 1u)) {
          ++pdone;
          prog = true;
        }
        if (np < pdone) {
          const bool first = np == 0 || pc.j == 0;
          const int sg = pseg + (first ? 1 : 0);
          if ((!first || sg == 0 || mbar_test_wait(ofree, uint32_t(sg - 1) & 1u)) &&
              mbar_test_wait(vfull(np & 1), uint32_t(np >> 1) & 1u)) {
            mma_pv(np, first);
            pseg = sg;
            ++np;
            tile_next(pc, s_prefix, B, U);
            prog = true;
          }
        }
        if (ns < cnt && pdone + 1 >= ns) {
          const bool first = ns == 0 || sc.j == 0;
          const int sg = sseg + (first ? 1 : 0);
          if ((!first || mbar_test_wait(qfull(sg & 1), uint32_t(sg >> 1) & 1u)) &&
              mbar_test_wait(kfull(ns & 1), uint32_t(ns >> 1) & 1u)) {
            mma_s(ns, sg & 1);
            sseg = sg;
            ++ns;
            tile_next(sc, s_prefix, B, U);
            prog = true;
          }
        }
        if (prog) {
          idle = 0;
        } else {  // bounded like every other wait: give up on a timeout or another abort
          if (idle == 0) t_idle = global_timer_ns();
          if ((++idle & 63u) == 0u) {
            if (*abort_flag) break;
            if (global_timer_ns() - t_idle > p.timeout_ns) {
              *abort_flag = 1;
              break;
            }
          }
        }
      }
      tc::commit(mdone);  // every MMA issued must have completed before TMEM is freed
      mbar_wait_bounded(mdone, 0u, p.timeout_ns);
    }
    __syncwarp();
  } else if (cnt > 0 && ((warp >= 2 && warp <= 5) || (PAIR && warp >= 7))) {
    // ---------------- softmax warps: one query row per CS threads ----------------
    // A warp reaches only its own quarter of the TMEM lanes, and the exponentials of a
    // lane quarter run on one SM sub-partition. With CS = 2 (at most 64 rows) each
    // quarter holds 16 rows, each twice (A rows 32q + j and 32q + 16 + j carry the same
    // Q row): the two threads of a row take half of the tile's columns each, their P rows
    // are zero outside their half and their O and l rows add up to the row's.
    // Paired (PAIR, bf16 caches, D = 128): warps 7..10 reach the same lane quarters as
    // 2..5, and the two warps of a quarter take half of each row's columns, half of its
    // O columns and half of its Q and output chunks; they share the row maximum of each
    // tile through shared memory (one mbarrier per quarter), so both weight their half
    // against the same reference.
    static_assert(CS == 1 || (CS == 2 && !kTiles), "split rows: one row tile only");
    static_assert(!PAIR || CS == 1, "paired warps: one thread per row");
    constexpr int kRpq = 32 / CS;                      // query rows per lane quarter
    constexpr int kNc = K::kN / CS / (PAIR ? 2 : 1);   // tile columns per thread
    constexpr int kOc = PAIR ? D / 2 : D;              // O columns of the row per thread
    const int quarter = warp & 3;  // warps 2, 3, 4, 5 own TMEM lanes 64.., 96.., 0.., 32..
                                   // (warps 7, 8, 9, 10: 96.., 0.., 32.., 64..)
    const int hp = PAIR && warp >= 7 ? 1 : 0;  // which half of the row (paired warps)
    const int sidx = warp >= 7 ? 128 + (warp - 7) * 32 + lane : tid - 64;  // 0.. softmax threads
    const int part = CS == 1 ? 0 : lane / kRpq;  // which kNc columns of the row it takes
    const int r = quarter * kRpq + lane % kRpq;  // query row of the unit
    const int ar = quarter * 32 + lane;          // A row / TMEM lane of this thread
    const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16);
    const float sl = p.scale_log2, asl = fabsf(sl);
    // this thread's query row of unit u: row (u % nsg) * R + r of its KV head (new
    // token Rg / g, query head Rg % g of the group), if it exists
    auto row_of = [&](int u) { return (u % nsg) * R + r; };
    auto row_exists = [&](int u) { return r < R && row_of(u) < rows; };
    TileCursor cur;
    tile_locate(cur, ra, s_prefix, B, U);
    // causal: new token i = Rg / g hides the last q_len - 1 - i positions of its head
    bool row_ok;
    int hide;
    if constexpr (kTiles) {
      row_ok = row_exists(cur.h);
      hide = row_ok ? p.q_len - 1 - row_of(cur.h) / p.g : 0;
    } else {
      row_ok = r < R;
      hide = row_ok ? p.q_len - 1 - r / p.g : 0;
    }
    // Q rows of the KV head at cursor t -> Q buffer qb (K-major, 128-byte swizzle), as
    // asynchronous copies (padding rows zero-filled); q_ready completes and publishes them
    auto prefetch_q = [&](const TileCursor& t, int qb) {
      constexpr int kChunks = D / 8;
      if (p.tma_out) {  // this warp's earlier output boxes have left these rows
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
      }
      const uint4* q = reinterpret_cast<const uint4*>(p.q);
      bool ex;
      size_t qrow;
      if constexpr (kTiles) {
        ex = row_exists(t.h);
        const int Rg = ex ? row_of(t.h) : 0;
        qrow = (size_t(t.s) * p.q_len + Rg / p.g) * p.Hq + (t.h / nsg) * p.g + Rg % p.g;
      } else {
        ex = row_ok;
        qrow = (size_t(t.s) * p.q_len + (ex ? r / p.g : 0)) * p.Hq + t.h * p.g +
               (ex ? r % p.g : 0);
      }
      const uint32_t qa = base + K::kOffQ + qb * K::kTile;
      constexpr int kQc = PAIR ? kChunks / 2 : kChunks;  // chunks of the row it copies
#pragma unroll
      for (int c1 = 0; c1 < kQc; ++c1) {
        const int cc = hp * kQc + c1;
        cp_async16(qa + (cc >> 3) * K::kSlab + ar * 128 + (((cc & 7) ^ (ar & 7)) << 4),
                   q + qrow * kChunks + cc, ex ? 16u : 0u);
      }
      cp_async_commit();
    };
    auto q_ready = [&](int qb) {
      cp_async_wait_all();
      fence_proxy_async_smem();  // generic-proxy writes before the MMAs read them
      mbar_arrive(qfull(qb));
    };
    // a warp whose 32 rows are all padding computes nothing: its P and O rows feed
    // output rows that are never stored
    const bool warp_idle = quarter * kRpq >= R;
    // rows of a head's last block past its context may hold anything (even NaN): the
    // softmax warps zero them in the V tile before P.V reads it (weights there are 0)
    auto zero_v_tail = [&](int i, int L, int t0) -> bool {
      const int zr0 = L - t0, zr1 = min(K::kN, ((L + BS - 1) / BS) * BS - t0);
      if (zr0 >= zr1) return true;
      if (!__all_sync(0xffffffffu, tc::wait_or_abort(vfull(i & 1), uint32_t(i >> 1) & 1u,
                                                     p.timeout_ns, abort_flag)))
        return false;
      const uint32_t vb = base + K::kOffV + (i & 1) * K::kTile;
      for (int idx = sidx; idx < (zr1 - zr0) * (D / 8); idx += K::kSoftThreads) {
        const int rr = zr0 + idx / (D / 8), cc = idx % (D / 8);
        tc::sts128(vb + (cc >> 3) * K::kSlab + rr * 128 + (((cc & 7) ^ (rr & 7)) << 4),
                   make_uint4(0u, 0u, 0u, 0u));
      }
      fence_proxy_async_smem();
      return true;
    };
    float m_ref = -INFINITY;
    int seg = 0, seg_j0 = cur.j, seg_tile = 0;
    bool ok = true;
    prefetch_q(cur, 0);
    q_ready(0);
    for (int i = 0; i < cnt; ++i) {
      const int st = i & 1;
      const bool first = i == 0 || cur.j == 0;
      const bool last = i == cnt - 1 || cur.j == cur.n - 1;
      if (first && i > 0) {  // this Q was published before the previous epilogue
        seg_j0 = cur.j;
        seg_tile = 0;
        if constexpr (kTiles) {
          row_ok = row_exists(cur.h);
          hide = row_ok ? p.q_len - 1 - row_of(cur.h) / p.g : 0;
        }
      }
      if (last && i + 1 < cnt) {  // the next unit's Q rows, while this tile runs
        TileCursor nx = cur;
        tile_next(nx, s_prefix, B, U);
        prefetch_q(nx, (seg + 1) & 1);
      }
      const int L = s_len[cur.s];
      const int t0 = cur.j * K::kN;  // first token of the tile
      if (!__all_sync(0xffffffffu, tc::wait_or_abort(sfull(st), uint32_t(i >> 1) & 1u,
                                                     p.timeout_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // columns this row may see in the tile (context end, causal limit); padding rows
      // take the warp's largest count so that the warp runs one path
      const int vis_row = row_ok ? min(K::kN, L - hide - t0) : -1;
      const int vis_w = __reduce_max_sync(0xffffffffu, vis_row);
      const int vis = row_ok ? vis_row : vis_w;
      if (warp_idle) {  // no row of this warp is stored: only keep the barriers going
        if (!zero_v_tail(i, L, t0)) {
          ok = false;
          break;
        }
        if (i > 0 && !__all_sync(0xffffffffu, tc::wait_or_abort(ofull, uint32_t(i - 1) & 1u,
                                                                p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        mbar_arrive(pfull);
        ++seg_tile;
        if (last) {
          if (i + 1 < cnt) q_ready((seg + 1) & 1);
          if (!__all_sync(0xffffffffu, tc::wait_or_abort(ofull, uint32_t(i) & 1u,
                                                         p.timeout_ns, abort_flag))) {
            ok = false;
            break;
          }
          mbar_arrive(ofree);
          ++seg;
        }
        tile_next(cur, s_prefix, B, U);
        continue;
      }
      // this thread's columns c0 .. c0 + kNc - 1 of the tile's scores
      const int c0 = (PAIR ? hp : part) * kNc;
      uint32_t s[kNc];
      if constexpr (PAIR) {
        tc::tmem_ld64(trow + K::kColS + st * K::kN + c0, s);
      } else if constexpr (CS == 1) {
        tc::tmem_ld128(trow + K::kColS + st * K::kN, s);
      } else {
        uint32_t sa[K::kN];
        tc::tmem_ld128(trow + K::kColS + st * K::kN, sa);
#pragma unroll
        for (int t = 0; t < kNc; ++t) s[t] = part == 0 ? sa[t] : sa[t + kNc];
      }
      if constexpr (kQ8) {  // one-byte caches: each column times its K scale
        if (!__all_sync(0xffffffffu, tc::wait_or_abort(kscale(i), uint32_t(i >> 2) & 1u,
                                                       p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        const uint32_t ks = scale_area(true, i) + 4 * c0;
#pragma unroll
        for (int t = 0; t < kNc; t += 4) {
          const uint4 k4 = lds128(ks + 4 * t);  // the same address in the lanes of a part
          s[t] = __float_as_uint(__uint_as_float(s[t]) * __uint_as_float(k4.x));
          s[t + 1] = __float_as_uint(__uint_as_float(s[t + 1]) * __uint_as_float(k4.y));
          s[t + 2] = __float_as_uint(__uint_as_float(s[t + 2]) * __uint_as_float(k4.z));
          s[t + 3] = __float_as_uint(__uint_as_float(s[t + 3]) * __uint_as_float(k4.w));
        }
      }
      if (sl < 0.f) {  // a negative scale is carried by the scores' signs
#pragma unroll
        for (int t = 0; t < kNc; ++t) s[t] ^= 0x80000000u;
      }
      // warp-uniform: every row sees the whole tile (all tiles but a head's last, and
      // the last ones of causal rows), else columns past each row's limit are masked
      const bool full = __all_sync(0xffffffffu, vis >= K::kN);
      if (!full) {
#pragma unroll
        for (int t = 0; t < kNc; ++t)
          if (c0 + t >= vis) s[t] = 0xff800000u;  // -inf
      }
      // tile maximum: three-input max over eight independent chains (then over the
      // row's CS threads)
      float mx[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mx[j] = __uint_as_float(s[j]);
#pragma unroll
      for (int u = 0; u < (kNc - 8) / 2; ++u)
        mx[u & 7] = fmax3(mx[u & 7], __uint_as_float(s[8 + 2 * u]), __uint_as_float(s[9 + 2 * u]));
      float mt = asl * fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                             fmaxf(mx[6], mx[7]));
      if constexpr (CS == 2) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, kRpq));
      if constexpr (PAIR) {  // the partner warp's half: [tile % 2][half][row] fp32
        const uint32_t xa = base + K::kOffXmax + uint32_t(i & 1) * 1024 + uint32_t(ar) * 4;
        tc::sts32(xa + hp * 512, __float_as_uint(mt));
        mbar_arrive(xmax(quarter));
        if (!__all_sync(0xffffffffu, tc::wait_or_abort(xmax(quarter), uint32_t(i) & 1u,
                                                       p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        mt = fmaxf(mt, __uint_as_float(lds32(xa + (hp ^ 1) * 512)));
      }
      float alpha = 1.f;
      bool rescale = false;
      if (vis > 0 && mt > m_ref + 8.f) {
        alpha = fast_exp2(m_ref - mt);  // 0 while the row has seen nothing
        m_ref = mt;
        rescale = seg_tile > 0;
      }
      // weights 2^(scale * s - m) (packed fp32x2 FMAs), bf16 pairs (fp16 over one-byte
      // caches); their row sums come from the tensor cores (P times a ones tile, beside
      // P.V)
      uint32_t pk[kNc / 2];
      const float2 asl2 = make_float2(asl, asl), nm2 = make_float2(-m_ref, -m_ref);
      if (full) {
#pragma unroll
        for (int t = 0; t < kNc; t += 2) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[t]), __uint_as_float(s[t + 1])),
                                      asl2, nm2);
          pk[t / 2] = kQ8 ? pack_f16x2(fast_exp2(x.x), fast_exp2(x.y))
                          : pack_bf16x2(fast_exp2(x.x), fast_exp2(x.y));
        }
      } else {
#pragma unroll
        for (int t = 0; t < kNc; t += 2) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[t]), __uint_as_float(s[t + 1])),
                                      asl2, nm2);
          const float w0 = c0 + t < vis ? fast_exp2(x.x) : 0.f,
                      w1 = c0 + t + 1 < vis ? fast_exp2(x.y) : 0.f;
          pk[t / 2] = kQ8 ? pack_f16x2(w0, w1) : pack_bf16x2(w0, w1);
        }
      }
      if (!zero_v_tail(i, L, t0)) {
        ok = false;
        break;
      }
      // P.V of the previous tile must be complete before P is overwritten or O rescaled
      if (i > 0 && !__all_sync(0xffffffffu, tc::wait_or_abort(ofull, uint32_t(i - 1) & 1u,
                                                              p.timeout_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int c1 = 0; c1 < kOc; c1 += 32) {
          const int c2 = hp * kOc + c1;
          uint32_t o[32];
          tc::tmem_ld32(trow + K::kColO + c2, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::tmem_st32(trow + K::kColO + c2, o);
        }
        if (hp == 0)
          tc::tmem_st1(trow + K::kColL,
                       __float_as_uint(__uint_as_float(tc::tmem_ld1(trow + K::kColL)) * alpha));
      }
      // P (column pairs); with CS = 2 each thread writes its half and zeros in the other,
      // a paired warp only its half
      if constexpr (PAIR) {
        tc::tmem_st32(trow + K::kColP + hp * (kNc / 2), pk);
      } else {
#pragma unroll
        for (int c2 = 0; c2 < K::kN / 2; c2 += 32) {
          uint32_t w[32];
          constexpr int kHalf = kNc / 2;  // column pairs per thread
#pragma unroll
          for (int e = 0; e < 32; ++e)
            w[e] = (CS == 1 || part == c2 / kHalf) ? pk[c2 % kHalf + e] : 0u;
          tc::tmem_st32(trow + K::kColP + c2, w);
        }
      }
      tc::fence_before_sync();
      mbar_arrive(pfull);
      ++seg_tile;
      if (last) {
        // the next KV head's Q (prefetched during this tile) goes to the MMA thread
        // first, so its scores are computed while this epilogue runs
        if (i + 1 < cnt) q_ready((seg + 1) & 1);
        // ---- segment epilogue: the output (whole head) or a partial record ----
        if (!__all_sync(0xffffffffu, tc::wait_or_abort(ofull, uint32_t(i) & 1u, p.timeout_ns,
                                                       abort_flag))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const bool whole = seg_j0 == 0 && cur.j == cur.n - 1;
        const size_t slot = size_t(2 * c + (seg == 0 ? 0 : 1));
        // the sum of the weights (over the row's CS threads)
        const float l1 = __uint_as_float(tc::tmem_ld1(trow + K::kColL));
        const float l = CS == 1 ? l1 : l1 + __shfl_xor_sync(0xffffffffu, l1, kRpq);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if (whole) {
          // the bf16 rows go through this segment's Q buffer (its MMAs are complete),
          // each row in its own Q row's slots (16-byte chunk k in slab k / 8, position
          // (k % 8) ^ (row % 8)): no other warp writes there, not even a faster warp
          // already prefetching the next Q rows; then 16 lanes store one contiguous
          // 2*D-byte output row
          constexpr int kCh = D / 8;  // 16-byte chunks of an output row
          const uint32_t qbuf = base + K::kOffQ + (seg & 1) * K::kTile;
          auto slot_addr = [&](int row, int ch) {
            return qbuf + (ch >> 3) * K::kSlab + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
          };
          fence_proxy_async_smem();  // the MMAs' reads of the buffer before these writes
#pragma unroll
          for (int c1 = 0; c1 < kOc; c1 += 32) {
            const int c2 = hp * kOc + c1;
            uint32_t o[32];
            tc::tmem_ld32(trow + K::kColO + c2, o);
            if constexpr (CS == 2) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                o[e] = __float_as_uint(__uint_as_float(o[e]) +
                                       __uint_as_float(__shfl_xor_sync(0xffffffffu, o[e], kRpq)));
            }
            if (part == 0) {
#pragma unroll
              for (int e = 0; e < 32; e += 8)
                tc::sts128(slot_addr(ar, (c2 + e) / 8),
                           make_uint4(pack_bf16x2(__uint_as_float(o[e]) * inv,
                                                  __uint_as_float(o[e + 1]) * inv),
                                      pack_bf16x2(__uint_as_float(o[e + 2]) * inv,
                                                  __uint_as_float(o[e + 3]) * inv),
                                      pack_bf16x2(__uint_as_float(o[e + 4]) * inv,
                                                  __uint_as_float(o[e + 5]) * inv),
                                      pack_bf16x2(__uint_as_float(o[e + 6]) * inv,
                                                  __uint_as_float(o[e + 7]) * inv)));
            }
          }
          if (p.tma_out) {
            // one TMA box per new token (its g rows) and 64-column slab (a paired warp:
            // its half's slab); g divides the warp's kRpq rows (32, or 16 in a split tile)
            // and the row tile (gs) starts on a token, so a token's rows belong to this
            // warp and its box starts on an atom
            fence_proxy_async_smem();  // the staged rows, for the async proxy
            __syncwarp();
            if (lane == 0) {
              if constexpr (kTiles) {
                const int rt0 = (cur.h % nsg) * R;  // first row of the tile in the head
                const int nloc = min(R, rows - rt0);  // rows of the tile that exist
                const int i0 = quarter * 32 / p.g, i1 = min(nloc, quarter * 32 + 32) / p.g;
                for (int i = i0; i < i1; ++i)
#pragma unroll
                  for (int s1 = 0; s1 < (PAIR ? 1 : K::kSlabs); ++s1) {
                    const int sl = PAIR ? hp : s1;
                    tma_store_2d(&tmo, qbuf + sl * K::kSlab + (i * p.g) * 128, sl * 64,
                                 (cur.s * p.q_len + rt0 / p.g + i) * p.Hq + (cur.h / nsg) * p.g);
                  }
              } else {
                // rows quarter * kRpq .. + kRpq - 1, staged from A row quarter * 32 on
                const int i0 = quarter * kRpq / p.g,
                          i1 = min(p.q_len, (quarter * kRpq + kRpq) / p.g);
                for (int i = i0; i < i1; ++i)
#pragma unroll
                  for (int s1 = 0; s1 < (PAIR ? 1 : K::kSlabs); ++s1) {
                    const int sl = PAIR ? hp : s1;
                    tma_store_2d(&tmo,
                                 qbuf + sl * K::kSlab +
                                     (quarter * (32 - kRpq) + i * p.g) * 128,
                                 sl * 64, (cur.s * p.q_len + i) * p.Hq + cur.h * p.g);
                  }
              }
              bulk_commit();
            }
          } else {
            __syncwarp();
            // lane l's own output row, handed to the lanes that store it
            long long my_row;
            int nrows;
            if constexpr (kTiles) {
              const int Rg = row_ok ? row_of(cur.h) : 0;
              my_row = (long long)((size_t(cur.s) * p.q_len + Rg / p.g) * p.Hq +
                                   (cur.h / nsg) * p.g + Rg % p.g);
              // rows of this warp that exist (a partial last row tile ends early)
              nrows = min(32, min(R, rows - (cur.h % nsg) * R) - quarter * 32);
            } else {
              my_row = (long long)((size_t(cur.s) * p.q_len + (row_ok ? r / p.g : 0)) * p.Hq +
                                   cur.h * p.g + (row_ok ? r % p.g : 0));
              nrows = min(kRpq, R - quarter * kRpq);
            }
            constexpr int kChw = PAIR ? kCh / 2 : kCh;  // chunks of a row this warp stores
#pragma unroll 4
            for (int k2 = 0; k2 < kChw; ++k2) {
              const int idx = k2 * 32 + lane, rl = idx / kChw, ch = hp * kChw + idx % kChw;
              const long long orow2 = __shfl_sync(0xffffffffu, my_row, rl);
              if (rl < nrows)
                reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                         size_t(orow2) * D)[ch] =
                    lds128(slot_addr(quarter * 32 + rl, ch));
            }
          }
        } else {
#pragma unroll
          for (int c1 = 0; c1 < kOc; c1 += 32) {
            const int c2 = hp * kOc + c1;
            uint32_t o[32];
            tc::tmem_ld32(trow + K::kColO + c2, o);
            if constexpr (CS == 2) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                o[e] = __float_as_uint(__uint_as_float(o[e]) +
                                       __uint_as_float(__shfl_xor_sync(0xffffffffu, o[e], kRpq)));
            }
            if (row_ok && part == 0) {
              float4* dst = reinterpret_cast<float4*>(p.part_o + (slot * R + r) * D + c2);
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                dst[e / 4] = make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                                         __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
            }
          }
        }
        if (row_ok && !whole && part == 0 && hp == 0)
          reinterpret_cast<float2*>(p.part_ml)[slot * R + r] = make_float2(m_ref, l);
        if (!whole && p.fixup && quarter == 0 && lane == 0 && hp == 0) {  // tail fixup
          volatile int* e = s_cut + 5 * int(slot & 1);
          e[0] = cur.s;
          e[1] = cur.h;
          e[2] = cur.n;
          e[3] = cur.j - seg_j0 + 1;
          e[4] = 1;
        }
        tc::fence_before_sync();
        mbar_arrive(ofree);
        ++seg;
        m_ref = -INFINITY;
      }
      tile_next(cur, s_prefix, B, U);
    }
    (void)ok;
    if (p.tma_out && lane == 0) bulk_wait_all();  // output boxes complete before exit
    tc::fence_before_sync();
  } else if (kQ8 && cnt > 0 && warp >= 7) {
    // ---------------- converters: one-byte codes -> bf16 values ----------------
    const int ct = tid - 7 * 32;
    TileCursor cur;
    tile_locate(cur, ra, s_prefix, B, U);
    bool ok = true;
    for (int i = 0; i < cnt && ok; ++i) {
      const int st = i & 1;
      const uint32_t par = uint32_t(i >> 1) & 1u;
      const int valid = min(K::kN, s_len[cur.s] - cur.j * K::kN);  // rows of the context
      for (int kv = 0; kv < 2; ++kv) {
        // every converter takes part in every barrier: they agree on going on first
        const bool landed = __all_sync(
            0xffffffffu,
            tc::wait_or_abort(kv == 0 ? kstage(st) : vstage(st), par, p.timeout_ns, abort_flag));
        if (!converters_all(landed)) {
          ok = false;
          break;
        }
        // K: the codes themselves as bf16 (exact), the score MMA's other operand being
        // the bf16 q, and the softmax multiplies each score column by its K scale (fp32);
        // V: code x scale as fp16, whose 11-bit significand keeps it within 2^-12 of its
        // value (P.V then runs on fp16 weights)
        if constexpr (kQ8) {
          const uint32_t tile = base + (kv == 0 ? K::kOffK : K::kOffV) + st * K::kTile;
          if (kv == 0) {
            convert_codes<D, (kQ8 ? CODE : 0), false, false>(tile, scale_area(true, i), valid,
                                                             ct);
            // scales of rows past the context may hold anything: zero for the softmax
            if (ct >= valid) tc::sts32(scale_area(true, i) + 4 * ct, 0u);
          } else {
            convert_codes<D, (kQ8 ? CODE : 0), true, true>(tile, scale_area(false, i), valid,
                                                           ct);
          }
        }
        fence_proxy_async_smem();  // the 16-bit values, for the MMAs (async proxy)
        converters_sync();
        if (ct == 0) {
          mbar_arrive(kv == 0 ? kfull(st) : vfull(st));
          if (kv == 0) mbar_arrive(kscale(i));
        }
      }
      tile_next(cur, s_prefix, B, U);
    }
  }
  __syncthreads();
  if (*abort_flag && tid == 0 && p.status) atomicOr(p.status, 0x4);
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, K::kTmemCols);
  }
  // cut heads this CTA completes (the tile buffers are idle: every copy has landed,
  // every MMA and output store has completed)
  if (p.fixup && !*abort_flag)
    tc_tail_fixup<D, kTiles>(p, s_prefix, s_rs, s_cut, gbase + K::kOffQ, K::kThreads);
}

template <int D, int BS, bool kTiles, int CODE, int CS = 1, bool PAIR = false>
DecodeKernelInfo tc_info() {
  using K = TcDecode<D, BS, (CODE >= 0), PAIR>;
  DecodeKernelInfo info{};
  info.fn =
      reinterpret_cast<const void*>(&paged_decode_tc_kernel<D, BS, kTiles, CODE, CS, PAIR>);
  info.warps = K::kThreads / 32;
  info.stages = 2;
  info.warp_smem = K::kFixedSmem;  // per CTA, plus 12 * (B + 1)
  info.mma = 1;
  info.simt_heads = 0;
  info.coop = 0;
  info.blk = 1;
  info.tc = 1;
  return info;
}

// row_tiles: several row tiles per KV head; split (one tile of at most 64 rows): two
// threads per query row, each with half of a tile's columns. Units of more than 64 rows
// over bf16 caches with D = 128 take two softmax warps per lane quarter (paired).
template <int CODE>
bool select_tc_code(int D, int BS, bool row_tiles, bool split, DecodeKernelInfo* info) {
  constexpr bool kPair = CODE < 0;
  if (row_tiles) {
    if (D == 128 && BS == 16) *info = tc_info<128, 16, true, CODE, 1, kPair>();
    else if (D == 128 && BS == 32) *info = tc_info<128, 32, true, CODE, 1, kPair>();
    else if (D == 64 && BS == 16) *info = tc_info<64, 16, true, CODE>();
    else if (D == 64 && BS == 32) *info = tc_info<64, 32, true, CODE>();
    else return false;
  } else if (split) {
    if (D == 128 && BS == 16) *info = tc_info<128, 16, false, CODE, 2>();
    else if (D == 128 && BS == 32) *info = tc_info<128, 32, false, CODE, 2>();
    else if (D == 64 && BS == 16) *info = tc_info<64, 16, false, CODE, 2>();
    else if (D == 64 && BS == 32) *info = tc_info<64, 32, false, CODE, 2>();
    else return false;
  } else {
    if (D == 128 && BS == 16) *info = tc_info<128, 16, false, CODE, 1, kPair>();
    else if (D == 128 && BS == 32) *info = tc_info<128, 32, false, CODE, 1, kPair>();
    else if (D == 64 && BS == 16) *info = tc_info<64, 16, false, CODE>();
    else if (D == 64 && BS == 32) *info = tc_info<64, 32, false, CODE>();
    else return false;
  }
  return true;
}

}  // namespace pkv
