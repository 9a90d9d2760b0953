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

__global__ void __launch_bounds__(128) paged_decode_merge_kernel(const MergeParams p) {
  pdl_wait_prior_grid();
  const int s = blockIdx.x / p.HU, u = blockIdx.x % p.HU;
  const int head0 = (u / p.nsg) * p.g + (u % p.nsg) * p.gs;
  const int n = p.prefix[s + 1] - p.prefix[s];
  const int tid = threadIdx.x;
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

  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  for (int i = tid; i < total; i += blockDim.x) {
    const int row = i / p.D, d = i % p.D;
    float M = -INFINITY;
    for (int w = w0; w <= w1; ++w) {
      const long long aw = worker_start(T, w, p.W);
      if (aw == worker_start(T, w + 1, p.W)) continue;
      const size_t slot = size_t(2 * w + ((w == w0 && aw != A) ? 1 : 0));
      M = fmaxf(M, ml[slot * p.gs + row].x);
    }
    float lsum = 0.f, acc = 0.f;
    for (int w = w0; w <= w1; ++w) {
      const long long aw = worker_start(T, w, p.W);
      if (aw == worker_start(T, w + 1, p.W)) continue;
      const size_t slot = size_t(2 * w + ((w == w0 && aw != A) ? 1 : 0));
      const float2 mlw = ml[slot * p.gs + row];
      const float f = fast_exp2(mlw.x - M);
      lsum += f * mlw.y;
      acc += f * p.part_o[(slot * p.gs + row) * p.D + d];
    }
    out[i] = __float2bfloat16_rn(acc / lsum);
  }
}

void launch_merge(const MergeParams& p, cudaStream_t stream) {
  const int grid = p.B * p.HU;
  if (grid <= 0) return;
  MergeParams copy = p;
  void* args[] = {&copy};
  launch_pdl(reinterpret_cast<const void*>(&paged_decode_merge_kernel), dim3(grid), dim3(128),
             args, 0, stream);
}

}  // namespace pkv
