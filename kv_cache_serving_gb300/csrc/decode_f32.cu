// decode_f32.cu -- fp32 KV instantiations of the decode kernels, the LSE merge,
// and the tiling queries the host uses to size chunks.
#include "decode.cuh"

namespace dsa {

cudaError_t launch_decode_f32(const DecodeLaunch& a, bool sparse, cudaStream_t s) {
  return sparse ? launch_decode_dispatch<float, true>(a, s)
                : launch_decode_dispatch<float, false>(a, s);
}

cudaError_t launch_merge(const DecodeLaunch& a, bool sparse, cudaStream_t s) {
  const int pairs = a.batch * a.hq;
  if (pairs == 0 || a.num_chunks <= 1) return cudaSuccess;
  const int blocks = (pairs + 3) / 4;
  if (a.head_dim == 64)
    sparse ? merge_kernel<64, true><<<blocks, 128, 0, s>>>(a)
           : merge_kernel<64, false><<<blocks, 128, 0, s>>>(a);
  else
    sparse ? merge_kernel<128, true><<<blocks, 128, 0, s>>>(a)
           : merge_kernel<128, false><<<blocks, 128, 0, s>>>(a);
  return cudaGetLastError();
}

int decode_rows_per_pass_f32(int head_dim, int group) {
  return decode_rows_per_pass_t<float>(head_dim, group);
}

int decode_ctas_per_sm_f32(int head_dim, int group, bool sparse) {
  return decode_ctas_per_sm_t<float>(head_dim, group, sparse);
}

}  // namespace dsa
