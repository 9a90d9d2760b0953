// append.cu -- write new tokens' K/V into their paged-cache slots.
//
// The block manager of "大模型工程（五）：推理优化核心技法" (chenk.top, section "块管理器：
// 分页如何运作") grows a request by appending physical blocks to its table; each new
// token then lands at slot = block * block_size + offset. The bf16 kernel is a pure
// scatter with 16-byte vector copies (one thread per 16-byte chunk). The INT8 kernel applies the
// per-(token, KV head) symmetric quantiser of section 2.3 of the gsyq.cn page with the
// round(w / s) form of "INT8 仅权重量化" (chenk.top): s = absmax / 127 and
// q = clamp(rint(x / s), -127, 127), both divisions IEEE round-to-nearest.
#include "common.cuh"
#include "internal.h"

namespace pkv {

// One thread copies one 16-byte chunk of one (token, KV head) row of K and of V.
__global__ void __launch_bounds__(256)
    paged_kv_append_bf16_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                uint4* __restrict__ kc, uint4* __restrict__ vc,
                                const int64_t* __restrict__ slots, int T, int Hkv, int D, int BS,
                                int NB) {
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const int cpr = D / 8;  // 16-byte chunks per head row
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)T * Hkv * cpr) return;
  const int t = int(i / (Hkv * cpr));
  const int rem = int(i % (Hkv * cpr));
  const int h = rem / cpr, dc = rem % cpr;
  const long long slot = slots[t];
  if (slot < 0 || slot >= (long long)NB * BS) return;
  const long long blk = slot / BS, off = slot % BS;
  const size_t dst = ((size_t(blk) * Hkv + h) * BS + off) * cpr + dc;
  kc[dst] = k[i];
  vc[dst] = v[i];
}

// One warp quantises one (token, KV head) row of K or V (blockIdx.y selects which).
template <int D>
__global__ void __launch_bounds__(128)
    paged_kv_append_int8_kernel(const __nv_bfloat16* __restrict__ k,
                                const __nv_bfloat16* __restrict__ v, int8_t* __restrict__ kc,
                                int8_t* __restrict__ vc, float* __restrict__ ks,
                                float* __restrict__ vs, const int64_t* __restrict__ slots, int T,
                                int Hkv, int BS, int NB) {
  constexpr int E = D / 32;  // elements per lane
  pdl_wait_prior_grid();
  pdl_allow_next_grid();
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= T * Hkv) return;
  const int t = row / Hkv, h = row % Hkv;
  const long long slot = slots[t];
  if (slot < 0 || slot >= (long long)NB * BS) return;
  const long long blk = slot / BS, off = slot % BS;
  const bool isv = blockIdx.y != 0;
  const __nv_bfloat16* src = (isv ? v : k) + size_t(row) * D + lane * E;
  float x[E];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    x[e] = __bfloat162float(src[e]);
    amax = fmaxf(amax, fabsf(x[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.0f);
  const size_t dst_row = (size_t(blk) * Hkv + h) * BS + off;
  int8_t* dst = (isv ? vc : kc) + dst_row * D + lane * E;
  int8_t q[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    int qi = 0;
    if (s > 0.f) qi = max(-127, min(127, __float2int_rn(__fdiv_rn(x[e], s))));
    q[e] = int8_t(qi);
  }
  if constexpr (E == 4) {
    *reinterpret_cast<char4*>(dst) = make_char4(q[0], q[1], q[2], q[3]);
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = q[e];
  }
  if (lane == 0) (isv ? vs : ks)[dst_row] = s;
}

cudaError_t launch_append_bf16(const void* k, const void* v, void* k_cache, void* v_cache,
                               const int64_t* slots, int T, int Hkv, int D, int BS, int NB,
                               cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const long long chunks = (long long)T * Hkv * (D / 8);
  const uint4* kk = static_cast<const uint4*>(k);
  const uint4* vv = static_cast<const uint4*>(v);
  uint4* kc = static_cast<uint4*>(k_cache);
  uint4* vc = static_cast<uint4*>(v_cache);
  void* args[] = {&kk, &vv, &kc, &vc, &slots, &T, &Hkv, &D, &BS, &NB};
  return launch_pdl(reinterpret_cast<const void*>(&paged_kv_append_bf16_kernel),
                    dim3(unsigned((chunks + 255) / 256)), dim3(256), args, 0, stream);
}

cudaError_t launch_append_int8(const void* k, const void* v, int8_t* k_cache, int8_t* v_cache,
                               float* k_scale, float* v_scale, const int64_t* slots, int T,
                               int Hkv, int D, int BS, int NB, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const dim3 grid((T * Hkv + 3) / 4, 2);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  void* args[] = {&kb, &vb, &k_cache, &v_cache, &k_scale, &v_scale, &slots, &T, &Hkv, &BS, &NB};
  const void* fn = D == 128 ? reinterpret_cast<const void*>(&paged_kv_append_int8_kernel<128>)
                 : D == 64  ? reinterpret_cast<const void*>(&paged_kv_append_int8_kernel<64>)
                            : nullptr;
  if (!fn) return cudaErrorInvalidValue;
  return launch_pdl(fn, grid, dim3(128), args, 0, stream);
}

}  // namespace pkv
