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

// Four codes (one 32-bit word, pre-processed by Codec::pre) times a scale -> two 16-bit
// pairs (bf16, or fp16 when kF16); zero when !live.
template <int CODE, bool kF16, bool kScale>
__device__ __forceinline__ void convert_word(uint32_t w, float sc, bool live, uint32_t& lo,
                                             uint32_t& hi) {
  using Codec = Code8<CODE>;
  const uint32_t b = Codec::pre(w);
  float2 f01 = unpack_f16x2(Codec::lo(b)), f23 = unpack_f16x2(Codec::hi(b));
  if constexpr (kScale) {
    f01.x *= sc;
    f01.y *= sc;
    f23.x *= sc;
    f23.y *= sc;
  }
  if constexpr (kF16) {
    lo = live ? pack_f16x2(f01.x, f01.y) : 0u;
    hi = live ? pack_f16x2(f23.x, f23.y) : 0u;
  } else {
    lo = live ? pack_bf16x2(f01.x, f01.y) : 0u;
    hi = live ? pack_bf16x2(f23.x, f23.y) : 0u;
  }
}

// One-byte codes of a 128-token tile -> 16-bit values (code x scale when kScale, one
// rounding; bf16, or fp16 when kF16) in the MMA layout of the tile's buffer (K-major,
// 128-byte swizzled 64-column slabs). The codes sit in the buffer's last kCodeTile
// bytes as the TMA wrote them (D-byte rows, 128- or 64-byte swizzle). Thread ct (0..127)
// converts token row ct: with D = 128 its codes occupy exactly the bytes its second
// slab row is written to, so it converts its first 64 columns (into slab 0, away from
// the codes), then reads the other 64 before writing them back over its own codes, and
// no thread waits for another; with D = 64 the rows of codes and of values do not line
// up, so every thread loads its codes, the converters meet, then write. Rows from
// `valid` on become zeros (their scales may hold anything).
template <int D, int CODE, bool kF16, bool kScale>
__device__ __forceinline__ void convert_codes(uint32_t tile, uint32_t scales, int valid,
                                              int ct) {
  constexpr int kN = 128, kSlab = kN * 128;
  constexpr int kSeg = D >= 128 ? 128 : 64;    // swizzle span of a row of codes
  const uint32_t stg = tile + uint32_t(D * 2 * kN - D * kN);
  const int t = ct;
  const bool live = t < valid;
  const float sc = kScale ? lds_f32(scales + 4 * t) : 1.f;
  const uint32_t out_row = tile + uint32_t(t * 128);
  // 16-byte chunk c (16 codes, columns 16c .. 16c + 15) -> value chunks 2 (c % 4) and
  // + 1 of slab c / 4
  auto write_chunk = [&](int c, const uint4& raw) {
    uint32_t o[8];
    convert_word<CODE, kF16, kScale>(raw.x, sc, live, o[0], o[1]);
    convert_word<CODE, kF16, kScale>(raw.y, sc, live, o[2], o[3]);
    convert_word<CODE, kF16, kScale>(raw.z, sc, live, o[4], o[5]);
    convert_word<CODE, kF16, kScale>(raw.w, sc, live, o[6], o[7]);
    const int ch0 = (c & 3) * 2;
    const uint32_t row = out_row + uint32_t((c >> 2) * kSlab);
    tc::sts128(row + uint32_t((ch0 ^ (t & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
    tc::sts128(row + uint32_t(((ch0 + 1) ^ (t & 7)) << 4), make_uint4(o[4], o[5], o[6], o[7]));
  };
  if constexpr (D == 128) {
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint4 raw[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        raw[k] = lds128(stg + swz<kSeg>(uint32_t(t * D + (4 * h + k) * 16)));
#pragma unroll
      for (int k = 0; k < 4; ++k) write_chunk(4 * h + k, raw[k]);
    }
  } else {
    uint4 raw[D / 16];
#pragma unroll
    for (int c = 0; c < D / 16; ++c) raw[c] = lds128(stg + swz<kSeg>(uint32_t(t * D + c * 16)));
    converters_sync();  // every read of the codes before any write over them
#pragma unroll
    for (int c = 0; c < D / 16; ++c) write_chunk(c, raw[c]);
  }
}

}  // namespace pkv
