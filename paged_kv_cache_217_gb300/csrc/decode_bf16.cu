// bf16 instantiations of the decode kernels.
#include "decode_launch.cuh"

namespace pkv {
cudaError_t launch_decode_bf16(const DecodeArgs& a, int head_dim, int gpad, cudaStream_t stream) {
  return launch_decode_t<__nv_bfloat16>(a, head_dim, gpad, stream);
}
}  // namespace pkv
