// decode_bf16.cu -- bf16 KV instantiations of the decode kernel for dense rows,
// and the bf16 entry points (the kept-list and fused modes' builds live in
// decode_bf16_list.cu and decode_bf16_mask.cu so that they compile in parallel).
#include "decode.cuh"

namespace dsa {

cudaError_t launch_decode_bf16_list(const DecodeLaunch& a, cudaStream_t s);
DecodeShape decode_shape_bf16_list(int head_dim, int group, int build);
cudaError_t launch_decode_bf16_mask(const DecodeLaunch& a, cudaStream_t s);
DecodeShape decode_shape_bf16_mask(int head_dim, int group, int build);

cudaError_t launch_decode_bf16(const DecodeLaunch& a, int mode, cudaStream_t s) {
  switch (mode) {
    case kRowsDense: return launch_decode_mode<bf16_t, kRowsDense>(a, s);
    case kRowsList: return launch_decode_bf16_list(a, s);
    case kRowsMask: return launch_decode_bf16_mask(a, s);
  }
  return cudaErrorInvalidValue;
}

DecodeShape decode_shape_bf16(int head_dim, int group, int mode, int build) {
  switch (mode) {
    case kRowsDense: return decode_shape_mode<bf16_t, kRowsDense>(head_dim, group, build);
    case kRowsList: return decode_shape_bf16_list(head_dim, group, build);
    case kRowsMask: return decode_shape_bf16_mask(head_dim, group, build);
  }
  return DecodeShape{0, 1, 1, DSA_DECODE_WARPS, 0, kBuildDefault};
}

}  // namespace dsa
