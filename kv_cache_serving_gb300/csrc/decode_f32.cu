// decode_f32.cu -- fp32 KV instantiations of the decode kernels, the LSE merge,
// and the tiling queries the host uses to size chunks.
#include "decode.cuh"

namespace dsa {

cudaError_t launch_decode_f32(const DecodeLaunch& a, int mode, cudaStream_t s) {
  switch (mode) {
    case kRowsDense: return launch_decode_mode<float, kRowsDense>(a, s);
    case kRowsList: return launch_decode_mode<float, kRowsList>(a, s);
    case kRowsMask: return launch_decode_mode<float, kRowsMask>(a, s);
  }
  return cudaErrorInvalidValue;
}

template <int D>
void launch_merge_d(const DecodeLaunch& a, int mode, int blocks, cudaStream_t s) {
  if (mode == kRowsDense) merge_kernel<D, kRowsDense><<<blocks, 128, 0, s>>>(a);
  else if (mode == kRowsList) merge_kernel<D, kRowsList><<<blocks, 128, 0, s>>>(a);
  else merge_kernel<D, kRowsMask><<<blocks, 128, 0, s>>>(a);
}

cudaError_t launch_merge(const DecodeLaunch& a, int mode, cudaStream_t s) {
  const int pairs = a.batch * a.hq;
  if (pairs == 0 || a.num_chunks <= 1) return cudaSuccess;
  const int blocks = (pairs + 3) / 4;
  if (a.head_dim == 64) launch_merge_d<64>(a, mode, blocks, s);
  else launch_merge_d<128>(a, mode, blocks, s);
  return cudaGetLastError();
}

DecodeShape decode_shape_f32(int head_dim, int group, int mode, int build) {
  switch (mode) {
    case kRowsDense: return decode_shape_mode<float, kRowsDense>(head_dim, group, build);
    case kRowsList: return decode_shape_mode<float, kRowsList>(head_dim, group, build);
    case kRowsMask: return decode_shape_mode<float, kRowsMask>(head_dim, group, build);
  }
  return DecodeShape{0, 1, 1, DSA_DECODE_WARPS, 0, kBuildDefault};
}

}  // namespace dsa
