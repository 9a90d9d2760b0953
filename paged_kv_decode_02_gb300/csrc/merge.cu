// merge.cu -- split-KV merge and finalize for paged decode.
//
// A (sequence, unit) whose blocks were cut between several decode workers left one
// unnormalised partial per worker: o_w = sum_t 2^(x_t - m_w) v_t, l_w = sum_t
// 2^(x_t - m_w), m_w = max_t x_t (scores x_t in log2 units). The exact softmax
// output is recovered with the online-softmax rescaling
//   m = max_w m_w,  l = sum_w 2^(m_w - m) l_w,  out = sum_w 2^(m_w - m) o_w / l.
// This kernel also writes zeros for empty sequences and, when a status word is
// given, validates each sequence's context length and block ids and zeroes the
// output of any sequence that fails.
#include "common.cuh"
#include "internal.h"

namespace pkv {

__device__ __forceinline__ long long worker_start(long long T, int w, int W) {
  return T * w / W;
}

// Largest worker w whose range [T*w/W, T*(w+1)/W) contains flat index x.
__device__ __forceinline__ int worker_of(long long x, long long T, int W) {
  return int(((x + 1) * W + T - 1) / T) - 1;
}

constexpr int kMergeThreads = 256;
constexpr int kMergeSlots = 1024;  // partial slots staged in shared memory per pass

__global__ void __launch_bounds__(kMergeThreads) paged_decode_merge_kernel(const MergeParams p) {
  pdl_wait_prior_grid();
  const int s = blockIdx.x / p.HU, u = blockIdx.x % p.HU;
  const int head0 = (u / p.nsg) * p.g + (u % p.nsg) * p.gs;
  const int n = p.prefix[s + 1] - p.prefix[s];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kMergeThreads / 32;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t(s) * p.Hq + head0) * p.D;
  const int total = p.gs * p.D;

  bool zero = (n == 0);
  if (p.status != nullptr) {
    __shared__ int bad;
    if (tid == 0) bad = 0;
    __syncthreads();
    int flags = 0;
    const int L = p.context_lens[s];
    if (tid == 0 && (L < 0 || L > p.MBS * p.BS)) flags |= 0x1;
    for (int j = tid; j < n; j += blockDim.x) {
      const int id = p.block_tables[size_t(s) * p.MBS + j];
      if (id < 0 || id >= p.NB) flags |= 0x2;
    }
    if (flags) atomicOr(&bad, flags);
    __syncthreads();
    if (bad) {
      if (tid == 0 && u == 0) atomicOr(p.status, bad);
      zero = true;
    }
  }
  if (zero) {
    for (int i = tid; i < total; i += blockDim.x) out[i] = __float2bfloat16_rn(0.f);
    return;
  }

  const long long T = (long long)p.HU * p.prefix[p.B];
  const long long A = (long long)p.HU * p.prefix[s] + (long long)u * n;
  const long long E = A + n;
  const int w0 = worker_of(A, T, p.W), w1 = worker_of(E - 1, T, p.W);
  if (w0 == w1) return;  // one worker covered the whole unit and wrote the output

  __shared__ int s_slot[kMergeSlots];
  __shared__ float s_max[16];
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  const int gs = p.gs, D = p.D;
  const int nq = total / 4;  // float4 outputs of this unit
  float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  float lsum[2] = {0.f, 0.f};

  // pass 1: the partial slots and each row's maximum over them
  const int P = w1 - w0 + 1;
  float rowmax = -INFINITY;  // lane-local, for row `warp` (+ kWarps)
  float rowmax2 = -INFINITY;
  for (int base = 0; base < P; base += kMergeSlots) {
    const int cnt = min(kMergeSlots, P - base);
    __syncthreads();
    for (int i = tid; i < cnt; i += blockDim.x) {
      const int w = w0 + base + i;
      const long long aw = worker_start(T, w, p.W);
      const bool empty = aw == worker_start(T, w + 1, p.W);
      s_slot[i] = empty ? -1 : 2 * w + ((w == w0 && aw != A) ? 1 : 0);
    }
    __syncthreads();
    for (int i = lane; i < cnt; i += 32) {
      const int slot = s_slot[i];
      if (slot < 0) continue;
      if (warp < gs) rowmax = fmaxf(rowmax, ml[size_t(slot) * gs + warp].x);
      if (warp + kWarps < gs) rowmax2 = fmaxf(rowmax2, ml[size_t(slot) * gs + warp + kWarps].x);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    rowmax = fmaxf(rowmax, __shfl_xor_sync(0xffffffffu, rowmax, o));
    rowmax2 = fmaxf(rowmax2, __shfl_xor_sync(0xffffffffu, rowmax2, o));
  }
  if (lane == 0) {
    if (warp < gs) s_max[warp] = rowmax;
    if (warp + kWarps < gs) s_max[warp + kWarps] = rowmax2;
  }

  // pass 2: rescale and sum (each thread owns up to two float4 outputs)
  for (int base = 0; base < P; base += kMergeSlots) {
    const int cnt = min(kMergeSlots, P - base);
    __syncthreads();
    if (P > kMergeSlots) {  // s_slot still holds the last chunk of pass 1: restage
      for (int i = tid; i < cnt; i += blockDim.x) {
        const int w = w0 + base + i;
        const long long aw = worker_start(T, w, p.W);
        const bool empty = aw == worker_start(T, w + 1, p.W);
        s_slot[i] = empty ? -1 : 2 * w + ((w == w0 && aw != A) ? 1 : 0);
      }
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int q = tid + k * kMergeThreads;
      if (q >= nq) break;
      const int row = (4 * q) / D, d = (4 * q) % D;
      const float M = s_max[row];
#pragma unroll 4
      for (int i = 0; i < cnt; ++i) {
        const int slot = s_slot[i];
        if (slot < 0) continue;
        const float2 mlw = ml[size_t(slot) * gs + row];
        const float f = fast_exp2(mlw.x - M);
        const float4 o = *reinterpret_cast<const float4*>(p.part_o + (size_t(slot) * gs + row) * D + d);
        lsum[k] += f * mlw.y;
        acc[k].x += f * o.x;
        acc[k].y += f * o.y;
        acc[k].z += f * o.z;
        acc[k].w += f * o.w;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int q = tid + k * kMergeThreads;
    if (q >= nq) break;
    const float inv = 1.f / lsum[k];
    uint2 pk;
    pk.x = pack_bf16x2(acc[k].x * inv, acc[k].y * inv);
    pk.y = pack_bf16x2(acc[k].z * inv, acc[k].w * inv);
    *reinterpret_cast<uint2*>(out + 4 * q) = pk;
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
