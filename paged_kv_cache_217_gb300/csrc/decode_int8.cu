// Decode over the INT8 KV cache. By default every group size runs the
// tensor-core INT8 tile (decode_mma_int8.cuh); PKV_INT8_MMA=0 selects the
// CUDA-core tile math with the int8 storage policy (decode.cuh, KvInt8),
// which needs no tensor maps and keeps V exact in fp32.
#include "decode_launch.cuh"
#include "decode_mma_int8.cuh"

#ifndef PKV_INT8_MMA
#define PKV_INT8_MMA 1
#endif

namespace pkv {
namespace {

// Stages per warp of the INT8 kernels (an int8 stage is half the size of a
// 16-bit one). The one-query tile (group size 1, head_dim <= 128: QK^T on
// dp4a, see mma_tile_int8_mha) takes kInt8MhaStages and 4 CTAs per SM (at
// most 128 registers): measured on GB300, the LLaMA-13B layer 87.1 -> 80.7 us
// against 4 stages at 3 CTAs per SM, the OPT-175B layer 670.6 -> 691.9 us.
constexpr int kInt8Stages = 4;
constexpr int kInt8MhaStages = 3;
// Warps per CTA of the INT8 tensor-core kernel for groups of 2..8 query
// heads (group size 1 keeps kGridWarps). Measured on GB300: the
// Llama-3-8B-shaped layer 39.1 us with 4 warps, 37.5 us with 3 (4 CTAs per
// SM); 3 warps for group size 1 made the LLaMA-13B layer 104.2 -> 113.7 us.
constexpr int kInt8GqaWarps = 3;
// One-query tile on one-pass grids of at most kLongGridCtas CTAs (few, long
// CTAs, see kLongGridWarps): 8 warps x kInt8MhaStages (2 CTAs per SM, the
// same 16 warps per SM), so the longest CTA streams at half its SM's rate
// instead of a quarter. Measured on GB300, OPT-175B layer over INT8 (768
// CTAs): 691.2-691.8 us with 4 x 3, 647.1-647.5 with 8 x 3, 649.2-649.3 with
// 8 x 2, 675.5 with 6 x 3, 677.1-677.2 with 6 x 4.
constexpr int kInt8LongWarps = 8;

template <typename T, int D, int G>
cudaError_t launch_int8_dg(const DecodeArgs& a, const CUtensorMap* kmap, const CUtensorMap* vmap,
                           cudaStream_t stream) {
  constexpr int NW = (PKV_INT8_MMA && G >= 2) ? kInt8GqaWarps : kGridWarps;
  constexpr int STAGES = (PKV_INT8_MMA && G == 1 && D <= 128) ? kInt8MhaStages : kInt8Stages;
  static bool configured[kMaxDevices] = {};
  // (the shared-prefix schedule: rows for its chunks, then the sequences, one pass)
  const dim3 grid(unsigned(a.num_kv_heads), unsigned(a.num_seqs + (a.prefix_header ? a.prefix_slots : 0)),
                  a.prefix_header ? 1u : unsigned(a.max_parts));
  cudaError_t err = cudaSuccess;
  if constexpr (PKV_INT8_MMA) {
    if constexpr (G == 1 && D <= 128) {
      const int64_t ctas = int64_t(grid.x) * grid.y * grid.z;
      if (grid.z == 1 && !a.prefix_header && ctas <= kLongGridCtas) {
        using CL = I8Cfg<D, kInt8LongWarps, kInt8MhaStages>;
        static_assert(CL::SMEM_BYTES <= 227 * 1024, "INT8 decode ring exceeds shared memory");
        auto kern = paged_decode_mma_int8_kernel<T, D, G, kInt8LongWarps, kInt8MhaStages>;
        static bool configured_long[kMaxDevices] = {};
        err = configure_once(kern, CL::SMEM_BYTES, configured_long);
        if (err != cudaSuccess) return err;
        err = launch_pdl(kern, grid, dim3(kInt8LongWarps * 32), CL::SMEM_BYTES, stream, a, *kmap, *vmap);
        if (err != cudaSuccess) return err;
        return cudaGetLastError();
      }
    }
    using C = I8Cfg<D, NW, STAGES>;
    static_assert(C::SMEM_BYTES <= 227 * 1024, "INT8 decode ring exceeds shared memory");
    auto kern = paged_decode_mma_int8_kernel<T, D, G, NW, STAGES>;
    err = configure_once(kern, C::SMEM_BYTES, configured);
    if (err != cudaSuccess) return err;
    err = launch_pdl(kern, grid, dim3(NW * 32), C::SMEM_BYTES, stream, a, *kmap, *vmap);
  } else {
    using C = DecodeCfg<T, D, G, NW, STAGES, KvInt8>;
    static_assert(C::SMEM_BYTES <= 227 * 1024, "INT8 decode ring exceeds shared memory");
    auto kern = paged_decode_kernel<T, D, G, NW, STAGES, KvInt8>;
    err = configure_once(kern, C::SMEM_BYTES, configured);
    if (err != cudaSuccess) return err;
    err = launch_pdl(kern, grid, dim3(NW * 32), C::SMEM_BYTES, stream, a);
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_int8_d(const DecodeArgs& a, int gpad, const CUtensorMap* kmap, const CUtensorMap* vmap,
                          cudaStream_t stream) {
  switch (gpad) {
    case 1: return launch_int8_dg<T, D, 1>(a, kmap, vmap, stream);
    case 2: return launch_int8_dg<T, D, 2>(a, kmap, vmap, stream);
    case 4: return launch_int8_dg<T, D, 4>(a, kmap, vmap, stream);
    case 8: return launch_int8_dg<T, D, 8>(a, kmap, vmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_int8_t(const DecodeArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                          const CUtensorMap* vmap, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_int8_d<T, 64>(a, gpad, kmap, vmap, stream);
    case 128: return launch_int8_d<T, 128>(a, gpad, kmap, vmap, stream);
    case 256: return launch_int8_d<T, 256>(a, gpad, kmap, vmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_int8_uses_tensor_maps() { return PKV_INT8_MMA != 0; }

cudaError_t launch_decode_int8(const DecodeArgs& a, bool bf16, int head_dim, int gpad, const CUtensorMap* kmap,
                               const CUtensorMap* vmap, cudaStream_t stream) {
  return bf16 ? launch_int8_t<__nv_bfloat16>(a, head_dim, gpad, kmap, vmap, stream)
              : launch_int8_t<__half>(a, head_dim, gpad, kmap, vmap, stream);
}

}  // namespace pkv
