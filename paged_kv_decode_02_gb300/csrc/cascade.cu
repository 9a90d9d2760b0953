// cascade.cu -- decode with a prefix shared by every sequence of the batch.
//
// Requests that share a prefix (a system prompt, few-shot examples: the prefix
// sharing of "分页注意力" in "大模型工程（五）：推理优化核心技法", chenk.top, and of
// section 2.2 of the gsyq.cn page) hold the same physical blocks at the head of their
// block tables. Every query row of a KV head then attends the same prefix keys, so for
// the prefix the B*g query rows of a KV head form a real dense contraction:
//   S = Q_rows (B*g x D) . K_prefix^T (D x P*bs),  O = softmax-weighted V_prefix.
// paged_prefix_kernel computes it once per KV head on the tensor cores (a producer warp
// streams each prefix block into shared memory once per CTA for four consumer warps of
// 16 query rows), leaving unnormalised partials per query row. The private suffixes go
// through the ordinary decode kernel (skipping the prefix entries of the tables), and
// paged_cascade_merge_kernel folds prefix and suffix partials with the online-softmax
// rescaling. The result equals decode attention over the whole table.
#include "decode.cuh"

namespace pkv {

template <int D, int BS, int kStages>
struct PrefixKernel {
  using Geo = TileGeom<false, D, BS>;
  static constexpr int kTile = Geo::kTileBytes;
  static constexpr int kConsumers = 4;                    // 16 query rows each
  static constexpr int kRows = 16 * kConsumers;
  static constexpr int kThreads = (kConsumers + 1) * 32;  // + one producer warp
  static constexpr int kOffV = kStages * kTile;
  static constexpr int kOffBar = 2 * kStages * kTile;     // full[kStages], empty[kStages]
  static constexpr int kSmem = kOffBar + 2 * kStages * 8 + 1024;
};

template <int D, int BS, int kStages>
__global__ void __launch_bounds__(PrefixKernel<D, BS, kStages>::kThreads)
    paged_prefix_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const PrefixParams pp) {
  using K = PrefixKernel<D, BS, kStages>;
  using Geo = typename K::Geo;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y, z = blockIdx.z;
  const int b0 = z * pp.per_split, b1 = min(pp.P, b0 + pp.per_split);
  const int nb = max(0, b1 - b0);
  auto sK = [&](int st) { return base + st * K::kTile; };
  auto sV = [&](int st) { return base + K::kOffV + st * K::kTile; };
  auto full = [&](int st) { return base + K::kOffBar + st * 8; };
  auto empty = [&](int st) { return base + K::kOffBar + (kStages + st) * 8; };
  pdl_wait_prior_grid();
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), K::kConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == K::kConsumers) {  // producer: one TMA stream per CTA
    if (lane == 0) {
      for (int i = 0; i < nb; ++i) {
        const int st = i % kStages;
        if (i >= kStages &&
            !mbar_wait_bounded(empty(st), uint32_t(i / kStages - 1) & 1u, pp.timeout_ns)) {
          if (pp.status) atomicOr(pp.status, 0x4);
          break;
        }
        int phys = __ldg(pp.prefix_ids + b0 + i);
        phys = (phys < 0 || phys >= pp.NB) ? 0 : phys;  // never copy outside the pool
        const int row = (phys * pp.Hkv + h) * BS;
        mbar_arrive_expect_tx(full(st), 2 * K::kTile);
#pragma unroll
        for (int hf = 0; hf < Geo::kHalves; ++hf) {
          const int x = hf * (Geo::kSeg / Geo::kElt);
          tma_load_2d(sK(st) + hf * BS * Geo::kSeg, &tmk, full(st), x, row);
          tma_load_2d(sV(st) + hf * BS * Geo::kSeg, &tmv, full(st), x, row);
        }
      }
    }
    return;
  }

  // consumer warp: query rows r0 = rbase + gid and r1 = r0 + 8 of KV head h
  MmaPathBf16<D, BS> path;
  path.init(lane);
  const int gid = lane >> 2;
  const int r0 = blockIdx.x * K::kRows + warp * 16 + gid, r1 = r0 + 8;
  const bool v0 = r0 < pp.R, v1 = r1 < pp.R;
  auto qrow = [&](int r) {
    const int s = r / pp.g, i = r % pp.g;
    return reinterpret_cast<const uint32_t*>(pp.q) + (size_t(s) * pp.Hq + h * pp.g + i) * (D / 2);
  };
  path.load_q(qrow(v0 ? r0 : 0), qrow(v1 ? r1 : 0), v0, v1);
  DecodeParams dp{};
  dp.scale_log2 = pp.scale_log2;
  for (int i = 0; i < nb; ++i) {
    const int st = i % kStages;
    if (!__all_sync(0xffffffffu,
                    mbar_wait_bounded(full(st), uint32_t(i / kStages) & 1u, pp.timeout_ns))) {
      if (lane == 0 && pp.status) atomicOr(pp.status, 0x4);
      return;
    }
    path.block(dp, sK(st), sV(st), 0u, 0u, BS);
    __syncwarp();
    if (lane == 0) {
      fence_proxy_async_smem();  // this warp's reads of the stage before the refill
      mbar_arrive(empty(st));
    }
  }
  const size_t rec = size_t(z * pp.Hkv + h) * pp.R;
  float2* ml = reinterpret_cast<float2*>(pp.pre_ml);
  path.store_rows(pp.pre_o + (rec + (v0 ? r0 : 0)) * D, pp.pre_o + (rec + (v1 ? r1 : 0)) * D,
                  ml + rec + (v0 ? r0 : 0), ml + rec + (v1 ? r1 : 0), v0, v1);
}

template <int D, int BS>
void prefix_info(const void** fn, int* smem) {
  constexpr int kStages = 4;
  *fn = reinterpret_cast<const void*>(&paged_prefix_kernel<D, BS, kStages>);
  *smem = PrefixKernel<D, BS, kStages>::kSmem;
}

bool select_prefix_kernel(int D, int BS, const void** fn, int* smem_bytes) {
  if (D == 128 && BS == 16) prefix_info<128, 16>(fn, smem_bytes);
  else if (D == 128 && BS == 32) prefix_info<128, 32>(fn, smem_bytes);
  else if (D == 64 && BS == 16) prefix_info<64, 16>(fn, smem_bytes);
  else if (D == 64 && BS == 32) prefix_info<64, 32>(fn, smem_bytes);
  else return false;
  return true;
}

// ---------------------------------------------------------------------------
// Cascade merge: one CTA per (sequence, unit) folds the nsplit prefix partials of its
// query rows and the suffix parts (the unit's own record when one decode worker
// covered the whole suffix, else the cut workers' slots). With a status word it first
// validates the sequence: context length in [prefix, max_blocks*block_size], block ids
// in the pool, and the table's head equal to the shared prefix (row 0); a sequence
// that fails gets a zero output.
// ---------------------------------------------------------------------------
constexpr int kCascadeThreads = 256;

__global__ void __launch_bounds__(kCascadeThreads)
    paged_cascade_merge_kernel(const CascadeMergeParams p) {
  pdl_wait_prior_grid();
  const int s = blockIdx.x / p.HU, u = blockIdx.x % p.HU;
  const int h = u / p.nsg, sg = u % p.nsg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gs = p.gs, D = p.D, Q = D / 4, nout = gs * Q;
  __nv_bfloat16* out =
      reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t(s) * p.Hq + h * p.g + sg * gs) * D;

  if (p.status != nullptr) {
    __shared__ int s_flags;
    if (tid == 0) s_flags = 0;
    __syncthreads();
    int flags = 0;
    const int L = p.context_lens[s];
    if (tid == 0 && (L < p.P * p.BS || L > p.MBS * p.BS)) flags |= (L < p.P * p.BS) ? 0x8 : 0x1;
    const int n = L <= 0 ? 0 : min((L + p.BS - 1) / p.BS, p.MBS);
    for (int j = tid; j < n; j += blockDim.x) {
      const int id = p.block_tables[size_t(s) * p.MBS + j];
      if (id < 0 || id >= p.NB) flags |= 0x2;
      if (j < p.P && id != p.block_tables[j]) flags |= 0x8;
    }
    if (flags) atomicOr(&s_flags, flags);
    __syncthreads();
    if (s_flags) {
      if (tid == 0 && u == 0) atomicOr(p.status, s_flags);
      for (int o = tid; o < nout; o += blockDim.x)
        *reinterpret_cast<uint2*>(out + size_t(o / Q) * D + 4 * (o % Q)) = make_uint2(0u, 0u);
      return;
    }
  }

  // the parts: nsplit prefix records, then the suffix parts
  // suffix parts: the decode kernel's flat order is (sequence, KV head, block) over Wg
  // workers of nsg warps; this unit's parts come from warp worker * nsg + sg
  const int n = p.prefix[s + 1] - p.prefix[s];
  const long long T = (long long)p.Hkv * p.prefix[p.B];
  const int Wg = p.Wg;
  int nsuf = 0, w0 = 0;
  bool dense = true, first_cut = false, whole = false;
  long long A = 0;
  if (n > 0) {
    A = (long long)p.Hkv * p.prefix[s] + (long long)h * n;
    w0 = int(((A + 1) * Wg + T - 1) / T) - 1;
    const int w1 = int(((A + n) * Wg + T - 1) / T) - 1;
    whole = (w0 == w1);
    dense = T >= Wg;
    nsuf = whole ? 1 : (dense ? (w1 - w0 + 1) : n);
    first_cut = (T * w0 / Wg) != A;
  }
  const int nparts = p.nsplit + nsuf;
  const size_t prow = size_t(s) * p.g + size_t(sg) * gs;  // prefix record row of row 0
  // row 0 of part i: (o, ml) base pointers
  auto part = [&](int i, const float*& o, const float2*& ml) {
    if (i < p.nsplit) {
      const size_t rec = size_t(i * p.Hkv + h) * p.R + prow;
      o = p.pre_o + rec * D;
      ml = reinterpret_cast<const float2*>(p.pre_ml) + rec;
      return;
    }
    const int k = i - p.nsplit;
    size_t slot;
    if (whole) slot = size_t(2 * p.W) + size_t(s) * p.HU + u;
    else if (dense) slot = size_t(2 * ((w0 + k) * p.nsg + sg) + ((k == 0 && first_cut) ? 1 : 0));
    else slot = size_t(2 * ((int(((A + k + 1) * Wg + T - 1) / T) - 1) * p.nsg + sg));
    o = p.part_o + slot * gs * D;
    ml = reinterpret_cast<const float2*>(p.part_ml) + slot * gs;
  };

  constexpr int kWarps = kCascadeThreads / 32;
  __shared__ float s_max[16];
  __shared__ float4 s_acc[kCascadeThreads];
  __shared__ float s_l[kCascadeThreads];
  for (int r = warp; r < gs; r += kWarps) {
    float mx = -INFINITY;
    for (int i = lane; i < nparts; i += 32) {
      const float* o;
      const float2* ml;
      part(i, o, ml);
      mx = fmaxf(mx, ml[r].x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) s_max[r] = mx;
  }
  __syncthreads();

  for (int o0 = 0; o0 < nout; o0 += blockDim.x) {
    const int span = min(nout - o0, int(blockDim.x));
    const int NG = blockDim.x / span;
    const int oi = o0 + tid % span, grp = tid / span;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (grp < NG) {
      const int row = oi / Q, dq = oi % Q;
      const float M = s_max[row];
      for (int i = grp; i < nparts; i += NG) {
        const float* o;
        const float2* ml;
        part(i, o, ml);
        const float2 v = ml[row];
        const float4 x = reinterpret_cast<const float4*>(o + size_t(row) * D)[dq];
        const float f = fast_exp2(v.x - M);
        L = fmaf(f, v.y, L);
        acc.x = fmaf(f, x.x, acc.x);
        acc.y = fmaf(f, x.y, acc.y);
        acc.z = fmaf(f, x.z, acc.z);
        acc.w = fmaf(f, x.w, acc.w);
      }
    }
    s_acc[tid] = acc;
    s_l[tid] = L;
    __syncthreads();
    if (grp == 0) {
      for (int k = 1; k < NG; ++k) {
        const float4 a = s_acc[k * span + (oi - o0)];
        acc.x += a.x;
        acc.y += a.y;
        acc.z += a.z;
        acc.w += a.w;
        L += s_l[k * span + (oi - o0)];
      }
      const float inv = 1.f / L;
      uint2 pk;
      pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(out + size_t(oi / Q) * D + 4 * (oi % Q)) = pk;
    }
    __syncthreads();
  }
}

void launch_cascade_merge(const CascadeMergeParams& p, cudaStream_t stream) {
  const int grid = p.B * p.HU;
  if (grid <= 0) return;
  CascadeMergeParams copy = p;
  void* args[] = {&copy};
  launch_pdl(reinterpret_cast<const void*>(&paged_cascade_merge_kernel), dim3(grid),
             dim3(kCascadeThreads), args, 0, stream);
}

}  // namespace pkv
