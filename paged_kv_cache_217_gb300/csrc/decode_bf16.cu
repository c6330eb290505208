// bf16 instantiations of the decode kernels.
#include "decode_launch.cuh"

namespace pkv {
cudaError_t launch_decode_bf16(const DecodeArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                              const CUtensorMap* vmap, cudaStream_t stream) {
  return launch_decode_t<__nv_bfloat16>(a, head_dim, gpad, kmap, vmap, stream);
}
cudaError_t launch_decode_sk_bf16(const SkArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                                 const CUtensorMap* vmap, cudaStream_t stream) {
  return launch_decode_sk_t<__nv_bfloat16>(a, head_dim, gpad, kmap, vmap, stream);
}
}  // namespace pkv
