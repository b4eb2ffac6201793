// decode_bf16_list.cu -- bf16 KV instantiations of the decode kernel that
// reads kept lists written by dsa_build_index (default and big-batch builds).
#include "decode.cuh"

namespace dsa {

cudaError_t launch_decode_bf16_list(const DecodeLaunch& a, cudaStream_t s) {
  return launch_decode_mode<bf16_t, kRowsList>(a, s);
}

DecodeShape decode_shape_bf16_list(int head_dim, int group, int build) {
  return decode_shape_mode<bf16_t, kRowsList>(head_dim, group, build);
}

}  // namespace dsa
