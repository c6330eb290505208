// Template dispatch of the decode kernels over head_dim and padded group size.
#pragma once

#include "decode.cuh"
#include "launch.h"

namespace pkv {

template <typename T, int D, int G>
cudaError_t launch_decode_dg(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int NW = 4;
  constexpr int STAGES = 2;
  using C = DecodeCfg<T, D, G, NW, STAGES>;
  auto kern = paged_decode_kernel<T, D, G, NW, STAGES>;
  static bool configured[kMaxDevices] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM_BYTES));
    if (err != cudaSuccess) return err;
    configured[dev] = true;
  }
  const dim3 grid(unsigned(a.num_kv_heads), unsigned(a.num_seqs), unsigned(a.max_parts));
  kern<<<grid, NW * 32, C::SMEM_BYTES, stream>>>(a);
  err = cudaGetLastError();
  if (err != cudaSuccess || a.max_parts <= 1) return err;
  const dim3 mgrid(unsigned(a.num_q_heads), unsigned(a.num_seqs));
  paged_decode_merge_kernel<T, D><<<mgrid, D, size_t(a.max_parts) * sizeof(float), stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_decode_d(const DecodeArgs& a, int gpad, cudaStream_t stream) {
  switch (gpad) {
    case 1: return launch_decode_dg<T, D, 1>(a, stream);
    case 2: return launch_decode_dg<T, D, 2>(a, stream);
    case 4: return launch_decode_dg<T, D, 4>(a, stream);
    case 8: return launch_decode_dg<T, D, 8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_decode_t(const DecodeArgs& a, int head_dim, int gpad, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_decode_d<T, 64>(a, gpad, stream);
    case 128: return launch_decode_d<T, 128>(a, gpad, stream);
    case 256: return launch_decode_d<T, 256>(a, gpad, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
