// decode_tc_e5m2.cu -- FP8 E5M2-cache instantiations of the tcgen05 decode kernel
// (decode_tc.cuh), in a unit of their own so that the kernels compile in parallel.
#include "decode_tc.cuh"

namespace pkv {

bool select_decode_tc_e5m2(int D, int BS, bool row_tiles, bool split,
                           DecodeKernelInfo* info) {
  return select_tc_code<CODE_E5M2>(D, BS, row_tiles, split, info);
}

}  // namespace pkv
