// decode_tc.cu -- bf16-cache instantiations of the tcgen05 decode kernel
// (decode_tc.cuh) and the kernel table over every KV dtype.
#include "decode_tc.cuh"

namespace pkv {

bool select_decode_tc(int D, int BS, bool row_tiles, bool split, int kvt,
                      DecodeKernelInfo* info) {
  switch (kvt) {
    case PKV_KV_BF16: return select_tc_code<-1>(D, BS, row_tiles, split, info);
    case PKV_KV_INT8: return select_decode_tc_int8(D, BS, row_tiles, split, info);
    case PKV_KV_FP8_E4M3: return select_decode_tc_e4m3(D, BS, row_tiles, split, info);
    case PKV_KV_FP8_E5M2: return select_decode_tc_e5m2(D, BS, row_tiles, split, info);
    default: return false;
  }
}

}  // namespace pkv
