// append.cu -- write new tokens' K/V into their paged-cache slots.
//
// The block manager of "大模型工程（五）：推理优化核心技法" (chenk.top, section "块管理器：
// 分页如何运作") grows a request by appending physical blocks to its table; each new
// token then lands at slot = block * block_size + offset. The bf16 kernel is a pure
// scatter with 16-byte vector copies (one thread per 16-byte chunk). The one-byte kernels
// apply the per-(token, KV head) symmetric quantiser of section 2.3 of the gsyq.cn page
// with the round(w / s) form of "INT8 仅权重量化" (chenk.top): s = absmax / 127 and
// q = clamp(rint(x / s), -127, 127), both divisions IEEE round-to-nearest; the FP8
// caches ("FP8（及 H100/H200 硬件路径）" and "KV 缓存量化", chenk.top: E4M3 or E5M2
// codes, per-token scales computed at run time) take s = absmax / 448 or / 57344 and
// round x / s to the nearest code, ties to even, saturating at the largest finite one.
#include <cuda_fp8.h>

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

// Code of x / s for each one-byte format. INT8: clamp(rint(x / s), -127, 127). FP8:
// the conversion instruction's round-to-nearest-even with saturation to the largest
// finite code (448 for E4M3, 57344 for E5M2). Both divisions are IEEE.
template <int CODE>
struct Encode8;
template <>
struct Encode8<CODE_I8> {
  static constexpr float kMax = 127.f;
  __device__ static __forceinline__ uint8_t code(float x, float s) {
    return uint8_t(int8_t(max(-127, min(127, __float2int_rn(__fdiv_rn(x, s))))));
  }
};
template <>
struct Encode8<CODE_E4M3> {
  static constexpr float kMax = 448.f;
  __device__ static __forceinline__ uint8_t code(float x, float s) {
    return uint8_t(__nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E4M3));
  }
};
template <>
struct Encode8<CODE_E5M2> {
  static constexpr float kMax = 57344.f;
  __device__ static __forceinline__ uint8_t code(float x, float s) {
    return uint8_t(__nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E5M2));
  }
};

// One warp quantises one (token, KV head) row of K or V (blockIdx.y selects which):
// s = absmax / kMax, code = Encode8(x, s); an all-zero row gets s = 0 and zero codes.
template <int D, int CODE>
__global__ void __launch_bounds__(128)
    paged_kv_append_q8_kernel(const __nv_bfloat16* __restrict__ k,
                              const __nv_bfloat16* __restrict__ v, uint8_t* __restrict__ kc,
                              uint8_t* __restrict__ vc, float* __restrict__ ks,
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
  const float s = __fdiv_rn(amax, Encode8<CODE>::kMax);
  const size_t dst_row = (size_t(blk) * Hkv + h) * BS + off;
  uint8_t* dst = (isv ? vc : kc) + dst_row * D + lane * E;
  uint8_t q[E];
#pragma unroll
  for (int e = 0; e < E; ++e) q[e] = s > 0.f ? Encode8<CODE>::code(x[e], s) : uint8_t(0);
  if constexpr (E == 4) {
    *reinterpret_cast<uchar4*>(dst) = make_uchar4(q[0], q[1], q[2], q[3]);
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

cudaError_t launch_append_q8(int code, const void* k, const void* v, void* k_cache,
                             void* v_cache, float* k_scale, float* v_scale, const int64_t* slots,
                             int T, int Hkv, int D, int BS, int NB, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const dim3 grid((T * Hkv + 3) / 4, 2);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  void* args[] = {&kb, &vb, &kc, &vc, &k_scale, &v_scale, &slots, &T, &Hkv, &BS, &NB};
  const void* fn = nullptr;
#define PKV_APPEND_Q8(DD, CC) \
  if (D == DD && code == CC) fn = reinterpret_cast<const void*>(&paged_kv_append_q8_kernel<DD, CC>);
  PKV_APPEND_Q8(128, CODE_I8)
  PKV_APPEND_Q8(64, CODE_I8)
  PKV_APPEND_Q8(128, CODE_E4M3)
  PKV_APPEND_Q8(64, CODE_E4M3)
  PKV_APPEND_Q8(128, CODE_E5M2)
  PKV_APPEND_Q8(64, CODE_E5M2)
#undef PKV_APPEND_Q8
  if (!fn) return cudaErrorInvalidValue;
  return launch_pdl(fn, grid, dim3(128), args, 0, stream);
}

}  // namespace pkv
