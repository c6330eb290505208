// Decode over the INT8 KV cache: the CUDA-core grid kernel with the int8
// storage format (codes and per-row scales staged together by the bulk-copy
// unit). The group is handled on CUDA cores for every group size: a tile of
// int8 codes is half the bytes of a 16-bit one, so the same per-warp pipeline
// reaches the HBM bound with fewer bytes in flight.
#include "decode_launch.cuh"

// Stages per warp of the INT8 kernel (an int8 stage is half the size of a
// 16-bit one, so twice as many give the same bytes in flight).
#ifndef PKV_INT8_STAGES
#define PKV_INT8_STAGES 4
#endif

namespace pkv {
namespace {

template <typename T, int D, int G>
cudaError_t launch_int8_dg(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int NW = PKV_GRID_WARPS;
  constexpr int STAGES = PKV_INT8_STAGES;
  using C = DecodeCfg<T, D, G, NW, STAGES, KvInt8>;
  static_assert(C::SMEM_BYTES <= 227 * 1024, "INT8 decode ring exceeds shared memory");
  auto kern = paged_decode_kernel<T, D, G, NW, STAGES, KvInt8>;
  static bool configured[kMaxDevices] = {};
  cudaError_t err = configure_once(kern, C::SMEM_BYTES, configured);
  if (err != cudaSuccess) return err;
  const dim3 grid(kSeqFastest ? unsigned(a.num_seqs) : unsigned(a.num_kv_heads),
                  kSeqFastest ? unsigned(a.num_kv_heads) : unsigned(a.num_seqs), unsigned(a.max_parts));
  err = launch_pdl(kern, grid, dim3(NW * 32), C::SMEM_BYTES, stream, a);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_int8_d(const DecodeArgs& a, int gpad, cudaStream_t stream) {
  switch (gpad) {
    case 1: return launch_int8_dg<T, D, 1>(a, stream);
    case 2: return launch_int8_dg<T, D, 2>(a, stream);
    case 4: return launch_int8_dg<T, D, 4>(a, stream);
    case 8: return launch_int8_dg<T, D, 8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_int8_t(const DecodeArgs& a, int head_dim, int gpad, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_int8_d<T, 64>(a, gpad, stream);
    case 128: return launch_int8_d<T, 128>(a, gpad, stream);
    case 256: return launch_int8_d<T, 256>(a, gpad, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_int8(const DecodeArgs& a, bool bf16, int head_dim, int gpad, cudaStream_t stream) {
  return bf16 ? launch_int8_t<__nv_bfloat16>(a, head_dim, gpad, stream)
              : launch_int8_t<__half>(a, head_dim, gpad, stream);
}

}  // namespace pkv
