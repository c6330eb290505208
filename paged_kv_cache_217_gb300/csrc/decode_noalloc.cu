// Decode attention without a caller-provided workspace.
//
// Split-K decode needs scratch memory for the partition partials. The regular
// entry point takes it from the caller. Some callers cannot allocate device
// memory when they decode: a serving engine that hands nearly all HBM to its
// KV-cache pool up front and has no room for ad-hoc allocations, or host code
// on a latency-critical path that must not call cudaMalloc/cudaFree (both can
// synchronise the device). This entry point serves them from a fixed scratch
// array that lives in the library's module memory: it allocates nothing.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "launch.h"
#include "paged_kv.h"
#include "status.h"

namespace {

// Fixed scratch shared by every call on a device. Every GPU that loads the
// library holds it until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// Device address of g_decode_scratch on the current device. In host code the
// symbol is only a host-side stand-in; the real address comes from
// cudaGetSymbolAddress, called once per device with that device current.
pkv_status_t scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[pkv::kMaxDevices] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (dev < 0 || dev >= pkv::kMaxDevices) return pkv::fail(PKV_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (err != cudaSuccess)
      return pkv::fail(PKV_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(err));
    addr[dev] = p;
  }
  *out = addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status_t pkv_paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int num_blocks, float scale, pkv_dtype_t dtype, int partition_size,
    pkv_stream_t stream) {
  void* scratch = nullptr;
  pkv_status_t st = scratch_address(&scratch);
  if (st != PKV_OK) return st;
  const size_t need = pkv_paged_attention_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                         max_blocks_per_seq, partition_size);
  if (need > size_t(PKV_NOALLOC_SCRATCH_BYTES))
    return pkv::fail(PKV_ERR_UNSUPPORTED,
                     "decode_noalloc: these sizes need %zu bytes of split-K scratch; the fixed scratch holds %zu "
                     "(use pkv_paged_attention_decode with a workspace, or a larger partition_size)",
                     need, size_t(PKV_NOALLOC_SCRATCH_BYTES));
  return pkv_paged_attention_decode(out, q, k_pool, v_pool, block_tables, context_lens, num_seqs, num_q_heads,
                                    num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype,
                                    partition_size, scratch, size_t(PKV_NOALLOC_SCRATCH_BYTES), stream);
}
