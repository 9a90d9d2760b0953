// decode_q8.cuh -- kernel choice for caches of one-byte codes with per-token scales
// (INT8, FP8 E4M3, FP8 E5M2); each code has its own translation unit.
#pragma once

#include "decode.cuh"

namespace pkv {

// CTA shape per path, from sweeps on GB300 with the INT8 cache: the tensor-core path
// (more arithmetic per byte) runs one warp per CTA with 12-16 KiB of stages; the
// CUDA-core path 8 warps with one ~8 KiB stage each.
template <int D, int BS>
struct Q8Shape {
  static constexpr int kStage = 2 * BS * D;  // K + V bytes of one block (scales aside)
  static constexpr int kMmaStages = kStage >= 8192 ? 2 : 12288 / kStage;
  static constexpr int kSimtStages = kStage >= 8192 ? 1 : 8192 / kStage;
};

template <int CODE, int D, int BS>
bool select_q8_shape(int simt_heads, DecodeKernelInfo* info, bool pair) {
  using S = Q8Shape<D, BS>;
  switch (simt_heads) {
    case 0:
      if constexpr (BS == 16) {
        if (pair) {  // 32-token items: two 16-token blocks per stage
          *info = make_decode_info<true, D, 16, MmaPathInt8<D, 32, CODE>, 1,
                                   Q8Shape<D, 32>::kMmaStages, false, 2>(1, 0);
          return true;
        }
      }
      *info = make_decode_info<true, D, BS, MmaPathInt8<D, BS, CODE>, 1, S::kMmaStages>(1, 0);
      return true;
    case 1:
      *info = make_decode_info<true, D, BS, SimtPath<true, D, BS, 1, CODE>, 8, S::kSimtStages>(
          0, 1);
      return true;
    case 2:
      *info = make_decode_info<true, D, BS, SimtPath<true, D, BS, 2, CODE>, 8, S::kSimtStages>(
          0, 2);
      return true;
    case 3:
      *info = make_decode_info<true, D, BS, SimtPath<true, D, BS, 3, CODE>, 8, S::kSimtStages>(
          0, 3);
      return true;
    default:
      return false;
  }
}

template <int CODE>
bool select_q8(int D, int BS, int simt_heads, DecodeKernelInfo* info, bool pair) {
  if (D == 128 && BS == 16) return select_q8_shape<CODE, 128, 16>(simt_heads, info, pair);
  if (D == 128 && BS == 32) return select_q8_shape<CODE, 128, 32>(simt_heads, info, pair);
  if (D == 64 && BS == 16) return select_q8_shape<CODE, 64, 16>(simt_heads, info, pair);
  if (D == 64 && BS == 32) return select_q8_shape<CODE, 64, 32>(simt_heads, info, pair);
  return false;
}

}  // namespace pkv
