// fp16 instantiations of the decode kernels.
#include "decode_launch.cuh"

namespace pkv {
cudaError_t launch_decode_f16(const DecodeArgs& a, int head_dim, int gpad, cudaStream_t stream) {
  return launch_decode_t<__half>(a, head_dim, gpad, stream);
}
}  // namespace pkv
