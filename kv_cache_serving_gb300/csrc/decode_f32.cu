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
cudaError_t launch_merge_d(const DecodeLaunch& a, int mode, int blocks, cudaStream_t s) {
  const dim3 grid(blocks), block(128);
  if (mode == kRowsDense) return launch_pdl(merge_kernel<D, kRowsDense>, grid, block, 0, s, a);
  if (mode == kRowsList) return launch_pdl(merge_kernel<D, kRowsList>, grid, block, 0, s, a);
  return launch_pdl(merge_kernel<D, kRowsMask>, grid, block, 0, s, a);
}

cudaError_t launch_merge(const DecodeLaunch& a, int mode, cudaStream_t s) {
  const int pairs = a.batch * a.hq;
  if (pairs == 0 || a.num_chunks <= 1) return cudaSuccess;
  const int blocks = (pairs + 3) / 4;
  return a.head_dim == 64 ? launch_merge_d<64>(a, mode, blocks, s)
                          : launch_merge_d<128>(a, mode, blocks, s);
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
