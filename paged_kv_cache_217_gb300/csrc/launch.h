// Host-side launchers of the CUDA kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace pkv {

struct DecodeArgs;
struct SkArgs;

constexpr int kMaxParts = 8192;   // split-K partitions per sequence (merge smem bound)
constexpr int kMaxDevices = 64;

// Decode. head_dim in {64,128,256}; gpad in {1,2,4,8}. gpad 1 runs the CUDA-core
// kernel; gpad >= 2 runs the tensor-core kernel, which reads the pools through
// the tensor maps kmap/vmap: three each, 128-byte swizzle, boxes of 16, 8 and
// 4 rows x 64 columns (the balanced schedule reads the first of each).
cudaError_t launch_decode_f16(const DecodeArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                              const CUtensorMap* vmap, cudaStream_t stream);
cudaError_t launch_decode_bf16(const DecodeArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                               const CUtensorMap* vmap, cudaStream_t stream);

// Decode with the balanced persistent schedule (decode_sk.cuh); same gpad rules.
cudaError_t launch_decode_sk_f16(const SkArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                                 const CUtensorMap* vmap, cudaStream_t stream);
cudaError_t launch_decode_sk_bf16(const SkArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                                  const CUtensorMap* vmap, cudaStream_t stream);

// Largest batch the balanced schedule takes for these sizes (its prefix sums
// share the CTA's shared memory with the rings); 0 for unsupported sizes.
int decode_sk_max_seqs(int head_dim, int gpad);

// The launch plan of a batch (num_seqs <= 1024) into `plan`: a 16-byte header
// {magic, num_seqs, 0, 0}, then the long-first order int32[num_seqs] (grid row
// -> sequence; the shortest sequences last with short_last); with `rows`, also
// int4[2 * num_seqs] per rank {sequence, length, ids 0..5 of `tables`} (the
// sequence -1 when tables is null).
cudaError_t launch_seq_order(const int32_t* lens, int num_seqs, int max_len, int window, bool short_last,
                             int4* plan, const int32_t* tables, int max_blocks, int4* rows, cudaStream_t stream);

// The prefix plan of the shared-prefix schedule (decode_prefix.cuh): header,
// groups int4[num_seqs / 2], chunks int4[num_seqs], the sequences outside any
// group int32[num_seqs], and the merge counters [num_seqs][num_kv_heads]
// zeroed. num_seqs <= 1024, tables of at most 256 blocks; groups of at most
// max_members sequences; slots = CTAs the decode grid holds at once.
cudaError_t launch_prefix_plan(const int32_t* lens, const int32_t* tables, int num_seqs, int max_blocks,
                               int num_kv_heads, int slots, int max_members, int4* header, int4* groups, int4* chunks,
                               int32_t* others, unsigned int* counters, cudaStream_t stream);
// CTAs of the shared-prefix decode grid (head_dim 64/128/256) resident at once on the current device.
cudaError_t prefix_resident_ctas(int head_dim, int* ctas);
// One warp that waits on an mbarrier no copy completes (bounded-wait self-test).
cudaError_t launch_bounded_wait_selftest(unsigned long long limit_ns, unsigned int* status, cudaStream_t stream);
cudaError_t launch_trace_stamp(unsigned long long* dst, cudaStream_t stream);

// Bit copies; element size is 2 bytes for both supported dtypes.
cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                                     const int64_t* slots, int num_tokens, int num_kv_heads,
                                     int head_dim, int num_blocks, unsigned int* status,
                                     cudaStream_t stream);
cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int64_t* pairs, int num_pairs,
                               int num_kv_heads, int head_dim, int num_blocks,
                               unsigned int* status, cudaStream_t stream);
// Block copy of two pools whose blocks are bytes_per_block bytes (a multiple of 16).
cudaError_t launch_copy_blocks_bytes(void* k_pool, void* v_pool, const int64_t* pairs, int num_pairs,
                                     int64_t bytes_per_block, int num_blocks, unsigned int* status,
                                     cudaStream_t stream);

// INT8 KV cache: quantising cache write (head_dim 64, 128 or 256) and decode
// over int8 codes with per-row fp32 scales. The tensor-core kernel reads the
// code pools through uint8 tensor maps (boxes of 16 rows x min(D, 128) bytes,
// 128-byte swizzle, 64-byte at D = 64); decode_int8_uses_tensor_maps() says
// whether the build needs them.
cudaError_t launch_reshape_and_cache_int8(const void* k, const void* v, bool bf16, int8_t* k_codes,
                                          int8_t* v_codes, float* k_scale, float* v_scale, const int64_t* slots,
                                          int num_tokens, int num_kv_heads, int head_dim, int num_blocks,
                                          unsigned int* status, cudaStream_t stream);
bool decode_int8_uses_tensor_maps();
cudaError_t launch_decode_int8(const DecodeArgs& a, bool bf16, int head_dim, int gpad, const CUtensorMap* kmap,
                               const CUtensorMap* vmap, cudaStream_t stream);

}  // namespace pkv
