// decode_bf16.cu -- bf16-cache instantiations of the paged decode kernel.
#include "decode.cuh"

namespace pkv {

namespace {
// Pipeline depth per warp keeps ~24 KiB of K+V tiles in flight per warp.
template <int D, int BS>
struct Bf16Shape {
  static constexpr int kTile = BS * D * 2;
  static constexpr int kWarps = (2 * kTile >= 16384) ? 3 : 4;
  static constexpr int kStagesRaw = 24576 / (2 * kTile);
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
};

template <int D, int BS>
bool select_shape(int simt_heads, DecodeKernelInfo* info) {
  using S = Bf16Shape<D, BS>;
  switch (simt_heads) {
    case 0:
      *info = make_decode_info<false, D, BS, MmaPathBf16<D, BS>, S::kWarps, S::kStages>(1, 0);
      return true;
    case 1:
      *info = make_decode_info<false, D, BS, SimtPath<false, D, BS, 1>, S::kWarps, S::kStages>(0, 1);
      return true;
    case 2:
      *info = make_decode_info<false, D, BS, SimtPath<false, D, BS, 2>, S::kWarps, S::kStages>(0, 2);
      return true;
    case 3:
      *info = make_decode_info<false, D, BS, SimtPath<false, D, BS, 3>, S::kWarps, S::kStages>(0, 3);
      return true;
    default:
      return false;
  }
}
}  // namespace

bool select_decode_bf16(int D, int BS, int simt_heads, DecodeKernelInfo* info) {
  if (D == 128 && BS == 16) return select_shape<128, 16>(simt_heads, info);
  if (D == 128 && BS == 32) return select_shape<128, 32>(simt_heads, info);
  if (D == 64 && BS == 16) return select_shape<64, 16>(simt_heads, info);
  if (D == 64 && BS == 32) return select_shape<64, 32>(simt_heads, info);
  return false;
}

}  // namespace pkv
