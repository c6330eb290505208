// C ABI entry points: host-side argument checks, partition choice, workspace
// sizing, the device status word, and dispatch to the kernel launchers.
// Semantics and citations of every call are in include/paged_kv.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "decode.cuh"
#include "launch.h"
#include "paged_kv.h"
#include "status.h"

namespace {

// Device status word: PKV_DEV_* flags raised by the kernels' index checks.
__device__ unsigned int g_pkv_status = 0u;

// Device address of g_pkv_status, looked up once per device with that device current.
pkv_status_t status_word(unsigned int** out) {
  static std::mutex mu;
  static unsigned int* addr[pkv::kMaxDevices] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (dev < 0 || dev >= pkv::kMaxDevices) return pkv::fail(PKV_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_pkv_status);
    if (err != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(err));
    addr[dev] = static_cast<unsigned int*>(p);
  }
  *out = addr[dev];
  return PKV_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int round_pow2_group(int g) {
  int p = 1;
  while (p < g) p <<= 1;
  return p;
}

// The library's partition choice. A CTA handles one partition of one
// (sequence, KV head); short contexts run in one pass, longer ones are split
// into 512-token partitions so that no CTA streams more than 32 tiles and
// long sequences spread over many SMs.
int choose_partition(int num_seqs, int num_kv_heads, int max_blocks_per_seq, int requested) {
  (void)num_seqs;
  (void)num_kv_heads;
  if (requested == -1) return -1;
  if (requested > 0) return requested;
  const int64_t max_ctx = int64_t(max_blocks_per_seq) * PKV_BLOCK_SIZE;
  if (max_ctx <= 512) return -1;
  return 512;
}

struct Plan {
  int part_tokens;  // tokens per partition as the kernel sees it
  int max_parts;
};

pkv_status_t plan_decode(int max_blocks_per_seq, int partition, Plan* plan) {
  const int64_t max_ctx = int64_t(max_blocks_per_seq) * PKV_BLOCK_SIZE;
  if (max_ctx > INT32_MAX / 2) return pkv::fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq too large");
  if (partition == -1) {
    plan->part_tokens = int(max_ctx);
    plan->max_parts = 1;
    return PKV_OK;
  }
  if (partition <= 0 || partition % PKV_BLOCK_SIZE != 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "partition_size must be 0, -1 or a positive multiple of 16 (got %d)", partition);
  const int64_t parts = (max_ctx + partition - 1) / partition;
  if (parts > pkv::kMaxParts)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "%lld partitions per sequence exceeds %d", (long long)parts, pkv::kMaxParts);
  plan->part_tokens = partition;
  plan->max_parts = int(parts);
  if (parts == 1) plan->part_tokens = int(max_ctx);  // one partition is one pass
  return PKV_OK;
}

size_t split_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_parts) {
  if (max_parts <= 1) return 0;
  const size_t rows = size_t(num_seqs) * size_t(num_q_heads) * size_t(max_parts);
  return rows * size_t(head_dim) * sizeof(float) + rows * sizeof(float2);
}

pkv_status_t cuda_status(cudaError_t err, const char* what) {
  if (err == cudaSuccess) return pkv::ok();
  return pkv::fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

bool supported_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

}  // namespace

extern "C" {

pkv_status_t pkv_device_status(uint32_t* flags_out, int clear) {
  if (!flags_out) return pkv::fail(PKV_ERR_INVALID_ARG, "device_status: flags_out is NULL");
  unsigned int* addr = nullptr;
  pkv_status_t st = status_word(&addr);
  if (st != PKV_OK) return st;
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return cuda_status(err, "cudaDeviceSynchronize");
  unsigned int v = 0;
  err = cudaMemcpy(&v, addr, sizeof(v), cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return cuda_status(err, "read status word");
  if (clear) {
    const unsigned int zero = 0;
    err = cudaMemcpy(addr, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (err != cudaSuccess) return cuda_status(err, "clear status word");
  }
  *flags_out = v;
  return pkv::ok();
}

int pkv_paged_attention_partition(int num_seqs, int num_kv_heads, int max_blocks_per_seq,
                                  int partition_size) {
  const int p = choose_partition(num_seqs, num_kv_heads, max_blocks_per_seq, partition_size);
  Plan plan;
  if (plan_decode(max_blocks_per_seq, p, &plan) != PKV_OK) return 0;
  return plan.max_parts <= 1 ? -1 : plan.part_tokens;
}

size_t pkv_paged_attention_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int max_blocks_per_seq,
                                          int partition_size) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  const int p = choose_partition(num_seqs, num_kv_heads, max_blocks_per_seq, partition_size);
  Plan plan;
  if (plan_decode(max_blocks_per_seq, p, &plan) != PKV_OK) return 0;
  return split_workspace_bytes(num_seqs, num_q_heads, head_dim, plan.max_parts);
}

pkv_status_t pkv_paged_attention_decode(void* out, const void* q, const void* k_pool,
                                        const void* v_pool, const int32_t* block_tables,
                                        const int32_t* context_lens, int num_seqs,
                                        int num_q_heads, int num_kv_heads, int head_dim,
                                        int max_blocks_per_seq, int num_blocks, float scale,
                                        pkv_dtype_t dtype, int partition_size, void* workspace,
                                        size_t workspace_bytes, pkv_stream_t stream) {
  if (num_seqs < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_seqs < 0");
  if (num_seqs == 0) return pkv::ok();
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                     num_q_heads, num_kv_heads);
  const int group = num_q_heads / num_kv_heads;
  if (group > 8) return pkv::fail(PKV_ERR_UNSUPPORTED, "query heads per KV head %d > 8", group);
  if (!supported_head_dim(head_dim)) return pkv::fail(PKV_ERR_UNSUPPORTED, "head_dim %d (64, 128 or 256)", head_dim);
  if (dtype != PKV_F16 && dtype != PKV_BF16) return pkv::fail(PKV_ERR_UNSUPPORTED, "dtype %d", int(dtype));
  if (max_blocks_per_seq <= 0 || num_blocks <= 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq and num_blocks must be > 0");
  if (num_seqs > 65535) return pkv::fail(PKV_ERR_UNSUPPORTED, "num_seqs %d > 65535", num_seqs);
  if (!std::isfinite(scale)) return pkv::fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens)
    return pkv::fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16))
    return pkv::fail(PKV_ERR_INVALID_ARG, "out, q, k_pool and v_pool must be 16-byte aligned");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4))
    return pkv::fail(PKV_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");

  const int p = choose_partition(num_seqs, num_kv_heads, max_blocks_per_seq, partition_size);
  Plan plan;
  pkv_status_t st = plan_decode(max_blocks_per_seq, p, &plan);
  if (st != PKV_OK) return st;
  const size_t need = split_workspace_bytes(num_seqs, num_q_heads, head_dim, plan.max_parts);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
    return pkv::fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) required, got %zu at %p",
                     need, workspace_bytes, workspace);

  unsigned int* status = nullptr;
  st = status_word(&status);
  if (st != PKV_OK) return st;

  pkv::DecodeArgs a;
  a.out = out;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.part_o = static_cast<float*>(workspace);
  a.part_ml = need > 0 ? reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                                   size_t(num_seqs) * num_q_heads * plan.max_parts *
                                                       head_dim * sizeof(float))
                       : nullptr;
  a.status = status;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.part_tokens = plan.part_tokens;
  a.max_parts = plan.max_parts;
  a.scale_log2 = scale * 1.4426950408889634f;

  const int gpad = round_pow2_group(group);
  cudaError_t err = dtype == PKV_F16 ? pkv::launch_decode_f16(a, head_dim, gpad, stream)
                                     : pkv::launch_decode_bf16(a, head_dim, gpad, stream);
  return cuda_status(err, "paged_attention_decode launch");
}

pkv_status_t pkv_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                                   const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                   int head_dim, int num_blocks, pkv_dtype_t dtype,
                                   pkv_stream_t stream) {
  if (num_tokens < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0) return pkv::ok();
  if (num_kv_heads <= 0 || num_blocks <= 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be > 0");
  if (head_dim <= 0 || head_dim % 8 != 0) return pkv::fail(PKV_ERR_UNSUPPORTED, "head_dim %d must be a multiple of 8", head_dim);
  if (dtype != PKV_F16 && dtype != PKV_BF16) return pkv::fail(PKV_ERR_UNSUPPORTED, "dtype %d", int(dtype));
  if (!k || !v || !k_pool || !v_pool || !slot_mapping) return pkv::fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(slot_mapping, 8))
    return pkv::fail(PKV_ERR_INVALID_ARG, "k, v and pools must be 16-byte aligned, slot_mapping 8-byte aligned");
  if (int64_t(num_tokens) * num_kv_heads * (head_dim / 8) > int64_t(UINT32_MAX) * 256)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "too many tokens for one launch");
  unsigned int* status = nullptr;
  pkv_status_t st = status_word(&status);
  if (st != PKV_OK) return st;
  return cuda_status(pkv::launch_reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, num_tokens,
                                                   num_kv_heads, head_dim, num_blocks, status, stream),
                     "reshape_and_cache launch");
}

pkv_status_t pkv_copy_blocks(void* k_pool, void* v_pool, const int64_t* src_dst_pairs,
                             int num_pairs, int num_kv_heads, int head_dim, int num_blocks,
                             pkv_dtype_t dtype, pkv_stream_t stream) {
  if (num_pairs < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_pairs < 0");
  if (num_pairs == 0) return pkv::ok();
  if (num_pairs > 65535) return pkv::fail(PKV_ERR_UNSUPPORTED, "num_pairs %d > 65535", num_pairs);
  if (num_kv_heads <= 0 || num_blocks <= 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be > 0");
  if (head_dim <= 0 || head_dim % 8 != 0) return pkv::fail(PKV_ERR_UNSUPPORTED, "head_dim %d must be a multiple of 8", head_dim);
  if (dtype != PKV_F16 && dtype != PKV_BF16) return pkv::fail(PKV_ERR_UNSUPPORTED, "dtype %d", int(dtype));
  if (!k_pool || !v_pool || !src_dst_pairs) return pkv::fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(src_dst_pairs, 8))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pools must be 16-byte aligned, pairs 8-byte aligned");
  unsigned int* status = nullptr;
  pkv_status_t st = status_word(&status);
  if (st != PKV_OK) return st;
  return cuda_status(pkv::launch_copy_blocks(k_pool, v_pool, src_dst_pairs, num_pairs, num_kv_heads,
                                             head_dim, num_blocks, status, stream),
                     "copy_blocks launch");
}

pkv_status_t pkv_check_copy_pairs(const int64_t* pairs, int num_pairs, int num_blocks) {
  if (num_pairs < 0 || num_blocks <= 0 || (num_pairs > 0 && !pairs))
    return pkv::fail(PKV_ERR_INVALID_ARG, "check_copy_pairs: bad argument");
  std::vector<char> is_src(size_t(num_blocks), 0), is_dst(size_t(num_blocks), 0);
  for (int i = 0; i < num_pairs; ++i) {
    const int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks)
      return pkv::fail(PKV_ERR_INVALID_ARG, "pair %d (%lld, %lld) outside [0, %d)", i, (long long)s, (long long)d, num_blocks);
    if (is_dst[size_t(d)]) return pkv::fail(PKV_ERR_INVALID_ARG, "block %lld is the dst of two pairs", (long long)d);
    is_dst[size_t(d)] = 1;
    is_src[size_t(s)] = 1;
  }
  for (int i = 0; i < num_pairs; ++i) {
    const int64_t d = pairs[2 * i + 1];
    if (is_src[size_t(d)]) return pkv::fail(PKV_ERR_INVALID_ARG, "block %lld is both a dst and a src", (long long)d);
  }
  return pkv::ok();
}

}  // extern "C"
