// convert.cuh -- one-byte KV codes widened to 16-bit MMA operands in shared memory, for
// the tcgen05 kernels (decode_tc.cuh, cascade.cu) over INT8 and FP8 caches.
//
// The quantised KV caches of "KV 缓存量化" (chenk.top page) hold one-byte codes and one
// fp32 scale per (token, KV head). The tensor-core kernels stream them as codes and
// widen them in shared memory: a tile's codes land (by TMA) in the last bytes of its
// 16-bit buffer, four converter warps (128 threads) widen them exactly (Code8) and write
// the 16-bit values over the whole buffer in the layout the MMA reads.
#pragma once

#include "decode.cuh"
#include "tcgen05.cuh"

namespace pkv {

// Named barrier of the four converter warps (id 1; __syncthreads uses 0).
__device__ __forceinline__ void converters_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
// The same barrier, returning whether v holds in every converter thread (so that the
// converters leave together when one of them gave up waiting).
__device__ __forceinline__ bool converters_all(bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred pv, pa; setp.ne.u32 pv, %1, 0; bar.red.and.pred pa, 1, 128, pv; "
      "selp.u32 %0, 1, 0, pa; }"
      : "=r"(r)
      : "r"(uint32_t(v))
      : "memory");
  return r != 0;
}

// One-byte codes of a 128-token tile -> 16-bit values (code x scale, one rounding; bf16,
// or fp16 when kF16) in the MMA layout of the tile's buffer (K-major, 128-byte swizzled
// 64-column slabs). The codes sit in the buffer's last kCodeTile bytes as the TMA wrote
// them (D-byte rows, 128- or 64-byte swizzle); every thread first loads all its chunks
// and scales, the converters meet, then write (the writes cover the codes). Rows from
// `valid` on become zeros (their scales may hold anything). ct: 0..127.
template <int D, int CODE, bool kF16, bool kScale>
__device__ __forceinline__ void convert_codes(uint32_t tile, uint32_t scales, int valid,
                                              int ct) {
  using Codec = Code8<CODE>;
  constexpr int kN = 128, kSlab = kN * 128;
  constexpr int kCh = D / 16;                  // 16-code chunks per row
  constexpr int kItems = kN * kCh / 128;       // chunks per thread
  constexpr int kSeg = D >= 128 ? 128 : 64;    // swizzle span of a row of codes
  const uint32_t stg = tile + uint32_t(D * 2 * kN - D * kN);
  uint4 raw[kItems];
  float sc[kItems];
#pragma unroll
  for (int m = 0; m < kItems; ++m) {
    const int item = ct + 128 * m, t = item / kCh, c = item % kCh;
    raw[m] = lds128(stg + swz<kSeg>(uint32_t(t * D + c * 16)));
    sc[m] = kScale ? lds_f32(scales + 4 * t) : 1.f;
  }
  converters_sync();  // every read of the codes before any write over them
#pragma unroll
  for (int m = 0; m < kItems; ++m) {
    const int item = ct + 128 * m, t = item / kCh, c = item % kCh;
    const uint32_t wd[4] = {raw[m].x, raw[m].y, raw[m].z, raw[m].w};
    uint32_t o[8];
    const bool live = t < valid;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t b = Codec::pre(wd[e]);
      const float2 f01 = unpack_f16x2(Codec::lo(b)), f23 = unpack_f16x2(Codec::hi(b));
      if constexpr (kF16) {
        o[2 * e] = live ? pack_f16x2(f01.x * sc[m], f01.y * sc[m]) : 0u;
        o[2 * e + 1] = live ? pack_f16x2(f23.x * sc[m], f23.y * sc[m]) : 0u;
      } else {
        o[2 * e] = live ? pack_bf16x2(f01.x * sc[m], f01.y * sc[m]) : 0u;
        o[2 * e + 1] = live ? pack_bf16x2(f23.x * sc[m], f23.y * sc[m]) : 0u;
      }
    }
    // columns 16c .. 16c + 15: slab 16c / 64, 16-byte chunks 2 (c % 4) and + 1 of it
    const int slab = (16 * c) >> 6, ch0 = ((16 * c) & 63) >> 3;
    const uint32_t row = tile + uint32_t(slab * kSlab + t * 128);
    tc::sts128(row + uint32_t(((ch0) ^ (t & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
    tc::sts128(row + uint32_t(((ch0 + 1) ^ (t & 7)) << 4), make_uint4(o[4], o[5], o[6], o[7]));
  }
}

}  // namespace pkv
