// decode_bf16.cu -- bf16 KV instantiations of the decode kernels.
#include "decode.cuh"

namespace dsa {

cudaError_t launch_decode_bf16(const DecodeLaunch& a, int mode, cudaStream_t s) {
  return launch_decode_t<bf16_t>(a, mode, s);
}

int decode_cluster_limit_bf16(int head_dim, int group) {
  return decode_cluster_limit_t<bf16_t>(head_dim, group);
}

int decode_rows_per_pass_bf16(int head_dim, int group) {
  return decode_rows_per_pass_t<bf16_t>(head_dim, group);
}

int decode_ctas_per_sm_bf16(int head_dim, int group, int mode) {
  return decode_ctas_per_sm_t<bf16_t>(head_dim, group, mode);
}

}  // namespace dsa
