// fp16 instantiations of the decode kernels.
#include "decode_launch.cuh"

namespace pkv {
cudaError_t launch_decode_f16(const DecodeArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                              const CUtensorMap* vmap, cudaStream_t stream) {
  return launch_decode_t<__half>(a, head_dim, gpad, kmap, vmap, stream);
}
cudaError_t launch_decode_sk_f16(const SkArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                                 const CUtensorMap* vmap, cudaStream_t stream) {
  return launch_decode_sk_t<__half>(a, head_dim, gpad, kmap, vmap, stream);
}
int decode_sk_max_seqs(int head_dim, int gpad) {
  // The limit depends only on sizes, not on the element type (both are 2 bytes).
  switch (head_dim) {
    case 64: return sk_max_seqs_d<__half, 64>(gpad);
    case 128: return sk_max_seqs_d<__half, 128>(gpad);
    case 256: return sk_max_seqs_d<__half, 256>(gpad);
    default: return 0;
  }
}
cudaError_t prefix_resident_ctas(int head_dim, int* ctas) {
  // fp16 and bf16 instantiations have the same shape and shared memory.
  switch (head_dim) {
    case 64: return prefix_resident_ctas_d<__half, 64>(ctas);
    case 128: return prefix_resident_ctas_d<__half, 128>(ctas);
    case 256: return prefix_resident_ctas_d<__half, 256>(ctas);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace pkv
