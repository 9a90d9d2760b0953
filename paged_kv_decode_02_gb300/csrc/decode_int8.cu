// decode_int8.cu -- INT8-cache instantiations of the paged decode kernel.
#include "decode.cuh"

namespace pkv {

namespace {
// CTA shape per path, from sweeps on GB300: the INT8 tensor-core path (more
// arithmetic per byte) runs one warp per CTA with 12-16 KiB of stages; the CUDA-core
// path 8 warps with one ~8 KiB stage each.
template <int D, int BS>
struct Int8Shape {
  static constexpr int kStage = 2 * BS * D;  // K + V bytes of one block (scales aside)
  static constexpr int kMmaStages = kStage >= 8192 ? 2 : 12288 / kStage;
  static constexpr int kSimtStages = kStage >= 8192 ? 1 : 8192 / kStage;
};

template <int D, int BS>
bool select_shape(int simt_heads, DecodeKernelInfo* info) {
  using S = Int8Shape<D, BS>;
  switch (simt_heads) {
    case 0:
      *info = make_decode_info<true, D, BS, MmaPathInt8<D, BS>, 1, S::kMmaStages>(1, 0);
      return true;
    case 1:
      *info = make_decode_info<true, D, BS, SimtPath<true, D, BS, 1>, 8, S::kSimtStages>(0, 1);
      return true;
    case 2:
      *info = make_decode_info<true, D, BS, SimtPath<true, D, BS, 2>, 8, S::kSimtStages>(0, 2);
      return true;
    case 3:
      *info = make_decode_info<true, D, BS, SimtPath<true, D, BS, 3>, 8, S::kSimtStages>(0, 3);
      return true;
    default:
      return false;
  }
}
}  // namespace

bool select_decode_int8(int D, int BS, int simt_heads, DecodeKernelInfo* info) {
  if (D == 128 && BS == 16) return select_shape<128, 16>(simt_heads, info);
  if (D == 128 && BS == 32) return select_shape<128, 32>(simt_heads, info);
  if (D == 64 && BS == 16) return select_shape<64, 16>(simt_heads, info);
  if (D == 64 && BS == 32) return select_shape<64, 32>(simt_heads, info);
  return false;
}

}  // namespace pkv
