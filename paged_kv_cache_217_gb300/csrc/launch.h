// Host-side launchers of the CUDA kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace pkv {

struct DecodeArgs;

constexpr int kMaxParts = 8192;   // split-K partitions per sequence (merge smem bound)
constexpr int kMaxDevices = 64;

// Decode (+ merge when a.max_parts > 1). head_dim in {64,128,256}; gpad in {1,2,4,8}.
cudaError_t launch_decode_f16(const DecodeArgs& a, int head_dim, int gpad, cudaStream_t stream);
cudaError_t launch_decode_bf16(const DecodeArgs& a, int head_dim, int gpad, cudaStream_t stream);

// Bit copies; element size is 2 bytes for both supported dtypes.
cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                                     const int64_t* slots, int num_tokens, int num_kv_heads,
                                     int head_dim, int num_blocks, unsigned int* status,
                                     cudaStream_t stream);
cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int64_t* pairs, int num_pairs,
                               int num_kv_heads, int head_dim, int num_blocks,
                               unsigned int* status, cudaStream_t stream);

}  // namespace pkv
