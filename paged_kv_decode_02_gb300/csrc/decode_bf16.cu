// decode_bf16.cu -- bf16-cache instantiations of the paged decode kernel (single-token
// and the causal multi-query variant).
#include "decode.cuh"

namespace pkv {

namespace {
// CTA shape per path, from sweeps on GB300 (the path is bound by per-warp latency, so
// more warps with shallow pipelines win): the CUDA-core path runs 8 warps per CTA with
// one ~8 KiB stage each (24 warps per SM at 16-token blocks); the tensor-core path 4
// warps with one stage. Larger tiles keep the per-warp bytes in flight near 8-16 KiB.
template <int D, int BS>
struct Bf16Shape {
  static constexpr int kStage = 2 * BS * D * 2;  // K + V bytes of one block
  static constexpr int kStages = kStage >= 8192 ? 1 : 8192 / kStage;
};
template <int D, int BS, bool MMA>
struct Bf16Warps {
  static constexpr int kWarps = MMA ? 4 : (Bf16Shape<D, BS>::kStage > 8192 ? 4 : 8);
};

template <int D, int BS>
bool select_shape(int simt_heads, DecodeKernelInfo* info, bool pair) {
  constexpr int kS = Bf16Shape<D, BS>::kStages;
  constexpr int kWm = Bf16Warps<D, BS, true>::kWarps, kWs = Bf16Warps<D, BS, false>::kWarps;
  switch (simt_heads) {
    case 0:
      if constexpr (BS == 16) {
        if (pair) {  // 32-token items: two 16-token blocks per stage
          *info = make_decode_info<false, D, 16, MmaPathBf16<D, 32>, kWm,
                                   Bf16Shape<D, 32>::kStages, false, 2>(1, 0);
          return true;
        }
      }
      *info = make_decode_info<false, D, BS, MmaPathBf16<D, BS>, kWm, kS>(1, 0);
      return true;
    case 1:
      *info = make_decode_info<false, D, BS, SimtPath<false, D, BS, 1>, kWs, kS>(0, 1);
      return true;
    case 2:
      *info = make_decode_info<false, D, BS, SimtPath<false, D, BS, 2>, kWs, kS>(0, 2);
      return true;
    case 3:
      *info = make_decode_info<false, D, BS, SimtPath<false, D, BS, 3>, kWs, kS>(0, 3);
      return true;
    default:
      return false;
  }
}
// Multi-query decode: workers of nsg warps share a ring of at least two stages (16 KiB
// or more in flight per worker). CTAs of 6 or 8 warps, whichever leaves fewer warps
// idle for the given nsg (at most one for nsg up to 8); on a tie the 6-warp CTA, two
// of which fit an SM (12 warps) where only one 8-warp CTA does.
template <int D, int BS>
struct MultiShape {
  static constexpr int kStage = Bf16Shape<D, BS>::kStage;
  static constexpr int kStages = kStage >= 8192 ? 2 : 16384 / kStage;
};
template <int D, int BS>
DecodeKernelInfo multi_shape(int nsg) {
  using Path = MmaPathBf16<D, BS, true>;
  constexpr int kS = MultiShape<D, BS>::kStages;
  const int idle6 = nsg <= 6 ? 6 % nsg : 6, idle8 = 8 % nsg;
  if (idle6 <= idle8) return make_decode_info<false, D, BS, Path, 6, kS, true>(1, 0);
  return make_decode_info<false, D, BS, Path, 8, kS, true>(1, 0);
}

// More than 8 row subgroups (over 128 rows per KV head): workers span CTAs, each warp
// with its own ring (4 warps per CTA, one stage).
template <int D, int BS>
DecodeKernelInfo multi_shape_wide() {
  return make_decode_info<false, D, BS, MmaPathBf16<D, BS, true>, Bf16Warps<D, BS, true>::kWarps,
                          Bf16Shape<D, BS>::kStages>(1, 0);
}
}  // namespace

bool select_decode_bf16_multi(int D, int BS, int nsg, DecodeKernelInfo* info) {
  if (nsg < 1) return false;
  const bool wide = nsg > 8;
  if (D == 128 && BS == 16) *info = wide ? multi_shape_wide<128, 16>() : multi_shape<128, 16>(nsg);
  else if (D == 128 && BS == 32) *info = wide ? multi_shape_wide<128, 32>() : multi_shape<128, 32>(nsg);
  else if (D == 64 && BS == 16) *info = wide ? multi_shape_wide<64, 16>() : multi_shape<64, 16>(nsg);
  else if (D == 64 && BS == 32) *info = wide ? multi_shape_wide<64, 32>() : multi_shape<64, 32>(nsg);
  else return false;
  return true;
}

bool select_decode_bf16(int D, int BS, int simt_heads, DecodeKernelInfo* info, bool pair) {
  if (D == 128 && BS == 16) return select_shape<128, 16>(simt_heads, info, pair);
  if (D == 128 && BS == 32) return select_shape<128, 32>(simt_heads, info, pair);
  if (D == 64 && BS == 16) return select_shape<64, 16>(simt_heads, info, pair);
  if (D == 64 && BS == 32) return select_shape<64, 32>(simt_heads, info, pair);
  return false;
}

}  // namespace pkv
