// decode_int8.cu -- INT8-cache instantiations of the paged decode kernel.
#include "decode_q8.cuh"

namespace pkv {

bool select_decode_int8(int D, int BS, int simt_heads, DecodeKernelInfo* info, bool pair) {
  return select_q8<CODE_I8>(D, BS, simt_heads, info, pair);
}

}  // namespace pkv
