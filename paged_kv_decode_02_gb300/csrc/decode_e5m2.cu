// decode_e5m2.cu -- FP8 E5M2-cache instantiations of the paged decode kernel.
#include "decode_q8.cuh"

namespace pkv {

bool select_decode_e5m2(int D, int BS, int simt_heads, DecodeKernelInfo* info, bool pair) {
  return select_q8<CODE_E5M2>(D, BS, simt_heads, info, pair);
}

}  // namespace pkv
