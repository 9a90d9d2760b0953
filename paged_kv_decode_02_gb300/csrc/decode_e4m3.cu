// decode_e4m3.cu -- FP8 E4M3-cache instantiations of the paged decode kernel.
#include "decode_q8.cuh"

namespace pkv {

bool select_decode_e4m3(int D, int BS, int simt_heads, DecodeKernelInfo* info, bool pair) {
  return select_q8<CODE_E4M3>(D, BS, simt_heads, info, pair);
}

}  // namespace pkv
