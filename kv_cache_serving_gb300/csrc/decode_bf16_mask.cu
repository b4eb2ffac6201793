// decode_bf16_mask.cu -- bf16 KV instantiations of the decode kernel that
// reads kept sets from the keep mask (both warps-per-CTA builds).
#include "decode.cuh"

namespace dsa {

cudaError_t launch_decode_bf16_mask(const DecodeLaunch& a, cudaStream_t s) {
  return launch_decode_mode<bf16_t, kRowsMask>(a, s);
}

DecodeShape decode_shape_bf16_mask(int head_dim, int group, int build) {
  return decode_shape_mode<bf16_t, kRowsMask>(head_dim, group, build);
}

}  // namespace dsa
