// merge.cu -- folds the partials of units cut between decode workers.
//
// A (sequence, unit) whose blocks were cut between several decode warps left one
// unnormalised partial per warp: o_w = sum_t 2^(x_t - m_w) v_t, l_w = sum_t
// 2^(x_t - m_w), m_w = max_t x_t (scores x_t in log2 units). The exact softmax output
// is recovered with the online-softmax rescaling
//   m = max_w m_w,  l = sum_w 2^(m_w - m) l_w,  out = sum_w 2^(m_w - m) o_w / l.
// One CTA per unit: it zero-fills empty sequences and, when a status word is given,
// validates the sequence's context length and block ids (zeroing the output of a
// sequence that fails); units the decode kernel finished itself then leave at once.
// The parts are shared out over thread groups so that a long context cut into many
// parts still merges in a few memory round trips.
#include "common.cuh"
#include "internal.h"

namespace pkv {

constexpr int kMergeThreads = 256;

__device__ __forceinline__ long long merge_worker_start(long long T, int w, int W) {
  return T * w / W;
}

// Largest worker w whose range [T*w/W, T*(w+1)/W) contains flat index x.
__device__ __forceinline__ int merge_worker_of(long long x, long long T, int W) {
  return int(((x + 1) * W + T - 1) / T) - 1;
}

__global__ void __launch_bounds__(kMergeThreads) paged_decode_merge_kernel(const MergeParams p) {
  pdl_wait_prior_grid();
  const int s = blockIdx.x / p.HU, u = blockIdx.x % p.HU;
  const int n = p.prefix[s + 1] - p.prefix[s];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gs = p.gs, D = p.D, Q = D / 4, nout = gs * Q;
  // output row of unit row r: (s * q_len + i) * Hq + kvh * g + j for the unit's query
  // row R = (u % nsg) * gs + r = i * g + j (with q_len = 1: head kvh * g + R)
  __nv_bfloat16* out_base = reinterpret_cast<__nv_bfloat16*>(p.out);
  auto out_row = [&](int r) -> __nv_bfloat16* {
    const int R = (u % p.nsg) * gs + r;
    return out_base + ((size_t(s) * p.q_len + R / p.g) * p.Hq + (u / p.nsg) * p.g + R % p.g) * D;
  };

  bool zero = (n == 0);
  if (p.status != nullptr) {
    __shared__ int s_flags;
    if (tid == 0) s_flags = 0;
    __syncthreads();
    int flags = 0;
    const int L = p.context_lens[s];
    if (tid == 0 && (L < 0 || L > p.MBS * p.BS || (L > 0 && L < p.q_len))) flags |= 0x1;
    for (int j = tid; j < n; j += blockDim.x) {
      const int id = p.block_tables[size_t(s) * p.MBS + j];
      if (id < 0 || id >= p.NB) flags |= 0x2;
    }
    if (flags) atomicOr(&s_flags, flags);
    __syncthreads();
    if (s_flags) {
      if (tid == 0 && u == 0) atomicOr(p.status, s_flags);
      zero = true;
    }
  }
  if (zero) {
    for (int o = tid; o < nout; o += blockDim.x)
      *reinterpret_cast<uint2*>(out_row(o / Q) + 4 * (o % Q)) = make_uint2(0u, 0u);
    return;
  }
  // the decode kernel's flat order is (sequence, KV head, block) over W workers of nsg
  // warps each; this unit's parts come from warp worker * nsg + sg of each worker
  const int nsg = p.nsg, kvh = u / nsg, sg = u % nsg, Hkv = p.HU / nsg;
  const long long T = (long long)Hkv * p.prefix[p.B];
  const long long A = (long long)Hkv * p.prefix[s] + (long long)kvh * n;
  const int W = p.W;
  const int w0 = merge_worker_of(A, T, W), w1 = merge_worker_of(A + n - 1, T, W);
  if (w0 == w1) return;  // one worker covered the whole unit and wrote the output
  // T >= W: every worker range is non-empty and the parts are workers w0..w1;
  // otherwise ranges hold one block at most and part i is the worker of block A + i
  const bool dense = T >= W;
  const int nparts = dense ? (w1 - w0 + 1) : n;
  const bool first_cut = merge_worker_start(T, w0, W) != A;
  auto slot_of = [&](int i) -> size_t {
    if (dense) return size_t(2 * ((w0 + i) * nsg + sg) + ((i == 0 && first_cut) ? 1 : 0));
    return size_t(2 * (merge_worker_of(A + i, T, W) * nsg + sg));
  };

  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  constexpr int kWarps = kMergeThreads / 32;
  __shared__ float s_max[16];
  __shared__ float4 s_acc[kMergeThreads];
  __shared__ float s_l[kMergeThreads];

  // pass 1: warp r finds the maximum of rows r and r + kWarps over the parts
  for (int r = warp; r < gs; r += kWarps) {
    float mx = -INFINITY;
    for (int i = lane; i < nparts; i += 32) mx = fmaxf(mx, ml[slot_of(i) * gs + r].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_max[r] = mx;
  }
  __syncthreads();

  // pass 2: thread (o, g) sums output float4 o over parts g, g + NG, ...
  for (int o0 = 0; o0 < nout; o0 += blockDim.x) {
  const int span = min(nout - o0, int(blockDim.x));
  const int NG = blockDim.x / span;
  const int o = o0 + tid % span, g = tid / span;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (g < NG) {
    const int row = o / Q, dq = o % Q;
    const float M = s_max[row] == -INFINITY ? 0.f : s_max[row];  // no part saw a token
#pragma unroll 4
    for (int i = g; i < nparts; i += NG) {
      const size_t slot = slot_of(i);
      const float2 v = ml[slot * gs + row];
      const float4 x = *(reinterpret_cast<const float4*>(p.part_o + (slot * gs + row) * D) + dq);
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
  if (g == 0) {
    for (int k = 1; k < NG; ++k) {
      const float4 a = s_acc[k * span + (o - o0)];
      acc.x += a.x;
      acc.y += a.y;
      acc.z += a.z;
      acc.w += a.w;
      L += s_l[k * span + (o - o0)];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;  // a row that saw nothing: zeros
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out_row(o / Q) + 4 * (o % Q)) = pk;
  }
  __syncthreads();  // s_acc is reused by the next span
  }
}

void launch_merge(const MergeParams& p, cudaStream_t stream) {
  const int grid = p.B * p.HU;
  if (grid <= 0) return;
  MergeParams copy = p;
  void* args[] = {&copy};
  launch_pdl(reinterpret_cast<const void*>(&paged_decode_merge_kernel), dim3(grid),
             dim3(kMergeThreads), args, 0, stream);
}

}  // namespace pkv
