// C ABI entry points: host-side argument checks, partition choice, workspace
// sizing, the device status word, and dispatch to the kernel launchers.
// Semantics and citations of every call are in include/paged_kv.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "decode.cuh"
#include "decode_sk.cuh"
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

constexpr int kBalanced = -2;  // partition choice: balanced persistent schedule
constexpr int kSharedPrefix = -5;  // partition choice: shared prompt prefixes read once per group
constexpr int64_t kLongFirstMaxCtas = 4096;  // grids up to ~9 waves start long sequences first

// CTAs the one-pass grid should have to keep every SM busy: 4 per SM of a
// 152-SM GB300 (3 are resident per SM; the fourth wave hides CTA start-up).
constexpr int64_t kFillCtas = 4 * 152;

// The library's schedule choice for partition_size == 0 (measured on GB300
// over the LLaMA-13B, Llama-3-8B, OPT-66B and OPT-175B layer workloads):
// one CTA per (sequence, KV head) whenever there are enough of them to fill
// the GPU -- it needs no merge and keeps sibling sequences that share prompt
// blocks in lockstep, so their reads hit L2. Too few (sequence, KV head)
// pairs are split into partitions just large enough to give kFillCtas CTAs
// (at least 256 tokens). The balanced persistent schedule (-2) is chosen
// only on request.
int choose_partition(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                     int requested) {
  (void)num_q_heads;
  (void)head_dim;
  if (requested == -1 || requested == kBalanced || requested == kSharedPrefix) return requested;
  if (requested > 0) return requested;
  const int64_t pairs = int64_t(num_seqs) * num_kv_heads;
  const int64_t max_ctx = int64_t(max_blocks_per_seq) * PKV_BLOCK_SIZE;
  if (pairs >= kFillCtas || max_ctx <= 256) return -1;
  const int64_t parts = (kFillCtas + pairs - 1) / pairs;
  int64_t p = (max_ctx + parts - 1) / parts;
  p = (p + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE * PKV_BLOCK_SIZE;
  if (p < 256) p = 256;
  return p >= max_ctx ? -1 : int(p);
}

// The long-first order (grid row -> sequence) of a batch is its launch plan.
// Batches of at least kOrderKernelMinSeqs sequences get it from a one-CTA
// kernel (seq_order_kernel) into the workspace instead of ranking the batch in
// every CTA, which costs each CTA a read of all the lengths and a CTA-wide
// ranking. Measured on GB300: Llama-3-8B layer (256 sequences) 44.5 -> 43.4 us,
// its INT8 cache 43.2 -> 41.3 us; on the 64-sequence LLaMA-13B layer the
// extra launch cost 0.9 %, so smaller batches rank in each CTA -- unless the
// caller made the plan beforehand (pkv_paged_attention_plan, once per decode
// step for all layers), which any batch of 2..1024 sequences can use.
constexpr int kOrderKernelMinSeqs = pkv::kRankInCtaMaxSeqs + 1;
bool long_first_grid(int num_seqs, int num_kv_heads, int max_parts) {
  return int64_t(num_seqs) * num_kv_heads * max_parts <= kLongFirstMaxCtas;
}
// Plan region of the workspace: a 16-byte header, int32[num_seqs] (the
// order, rounded up to 16 bytes), then int4[2 * num_seqs] of rows {sequence,
// length, block ids 0..5} in the order's ranks.
size_t plan_bytes(int num_seqs, int num_kv_heads, int max_parts) {
  if (num_seqs < 2 || num_seqs > pkv::kOrderMaxSeqs || !long_first_grid(num_seqs, num_kv_heads, max_parts)) return 0;
  return 16 + (size_t(num_seqs) * sizeof(int32_t) + 15) / 16 * 16 + size_t(num_seqs) * 32;
}
int4* plan_rows_of(int4* plan_hdr, int num_seqs) {
  if (!plan_hdr) return nullptr;
  return reinterpret_cast<int4*>(reinterpret_cast<char*>(plan_hdr) + 16 +
                                 (size_t(num_seqs) * sizeof(int32_t) + 15) / 16 * 16);
}

// Sizes the shared-prefix schedule takes: batches the plan kernel covers,
// tables it compares, and at least two members per group (query heads per KV
// head at most 4: a group's query rows fill at most kPrefixRows MMA rows).
bool prefix_fits(int num_seqs, int num_q_heads, int num_kv_heads, int max_blocks_per_seq) {
  const int group = num_kv_heads > 0 ? num_q_heads / num_kv_heads : 0;
  return group >= 1 && group <= pkv::kPrefixRows / 2 && num_seqs >= 2 && num_seqs <= pkv::kOrderMaxSeqs &&
         max_blocks_per_seq <= pkv::kPrefixMaxBlocks;
}
int prefix_max_members(int num_q_heads, int num_kv_heads) { return pkv::kPrefixRows / (num_q_heads / num_kv_heads); }

// Workspace of the shared-prefix schedule: the split-K layout with
// kPrefixMaxParts partitions (the partials of split groups, one arrival
// counter per (group's first sequence, KV head)), then the prefix plan:
// header int4, groups int4[num_seqs / 2], chunks int4[num_seqs], the
// sequences outside any group int32[num_seqs] (16-byte rounded).
struct PrefixLayout {
  size_t header_offset, groups_offset, chunks_offset, others_offset, total;
  int max_chunks;
};

PrefixLayout prefix_layout(size_t split_total, int num_seqs) {
  PrefixLayout l;
  const int max_groups = num_seqs / 2 > 0 ? num_seqs / 2 : 1;
  l.max_chunks = num_seqs;
  l.header_offset = split_total;
  l.groups_offset = l.header_offset + 16;
  l.chunks_offset = l.groups_offset + size_t(max_groups) * 16;
  l.others_offset = l.chunks_offset + size_t(l.max_chunks) * 16;
  l.total = l.others_offset + (size_t(num_seqs) * sizeof(int32_t) + 15) / 16 * 16;
  return l;
}

// CTAs of the shared-prefix grid resident at once on the current device, per
// head_dim (64, 128, 256), looked up once per device.
pkv_status_t prefix_slots(int head_dim, int* slots) {
  static std::mutex mu;
  static int cache[pkv::kMaxDevices][3] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= pkv::kMaxDevices)
    return pkv::fail(PKV_ERR_CUDA, "no usable current CUDA device");
  const int i = head_dim == 64 ? 0 : head_dim == 128 ? 1 : 2;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][i] <= 0) {
    int n = 0;
    const cudaError_t err = pkv::prefix_resident_ctas(head_dim, &n);
    if (err != cudaSuccess)
      return pkv::fail(PKV_ERR_CUDA, "occupancy of the shared-prefix grid: %s", cudaGetErrorString(err));
    cache[dev][i] = n > 0 ? n : 1;
  }
  *slots = cache[dev][i];
  return PKV_OK;
}

bool balanced_fits(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim) {
  const int group = num_kv_heads > 0 ? num_q_heads / num_kv_heads : 0;
  int gpad = 1;
  while (gpad < group) gpad <<= 1;
  return num_kv_heads < 512 && gpad <= 8 && num_seqs <= pkv::decode_sk_max_seqs(head_dim, gpad);
}

// Workspace of the balanced schedule: two partial slots per persistent warp
// (acc[group][D], m[group], l[group] in fp32, 16-byte rounded), then one
// arrival counter per (sequence, KV head).
struct SkLayout {
  int slot_floats;
  size_t counter_offset, counter_bytes, total;
};

SkLayout sk_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim) {
  SkLayout l;
  const int group = num_q_heads / num_kv_heads;
  l.slot_floats = (group * (head_dim + 2) + 3) / 4 * 4;
  l.counter_offset = size_t(2) * pkv::kSkMaxWarps * size_t(l.slot_floats) * sizeof(float);
  l.counter_bytes = size_t(num_seqs) * size_t(num_kv_heads) * sizeof(unsigned int);
  l.total = (l.counter_offset + l.counter_bytes + 15) / 16 * 16;
  return l;
}

struct Plan {
  int part_tokens;  // tokens per partition as the kernel sees it
  int max_parts;
};

pkv_status_t plan_decode(int max_blocks_per_seq, int partition, Plan* plan) {
  const int64_t max_ctx = int64_t(max_blocks_per_seq) * PKV_BLOCK_SIZE;
  if (max_ctx > INT32_MAX / 2) return pkv::fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq too large");
  if (partition == kBalanced) {
    plan->part_tokens = 0;
    plan->max_parts = 0;
    return PKV_OK;
  }
  if (partition == -1 || partition == kSharedPrefix) {
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

// Split-K workspace: part_o fp32 [S][Hq][P][D] | part_ml float2 [S][Hq][P] |
// counters u32 [S][Hkv] (partitions finished per (sequence, KV head)).
struct SplitLayout {
  size_t ml_offset, counter_offset, counter_bytes, total;
};

SplitLayout split_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_parts) {
  SplitLayout l{0, 0, 0, 0};
  if (max_parts <= 1) return l;
  const size_t rows = size_t(num_seqs) * size_t(num_q_heads) * size_t(max_parts);
  l.ml_offset = rows * size_t(head_dim) * sizeof(float);
  l.counter_offset = l.ml_offset + rows * sizeof(float2);
  l.counter_bytes = size_t(num_seqs) * size_t(num_kv_heads) * sizeof(unsigned int);
  l.total = (l.counter_offset + l.counter_bytes + 15) / 16 * 16;
  return l;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A pool [num_blocks][num_kv_heads][16][head_dim] seen as a 2-D tensor of
// num_blocks*num_kv_heads*16 rows by head_dim columns, read in boxes of
// box_rows (16, 8 or 4) rows x 64 columns with the 128-byte swizzle.
pkv_status_t pool_tensor_map(CUtensorMap* map, const void* pool, int64_t rows, int head_dim,
                             pkv_dtype_t dtype, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return pkv::fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cuuint64_t(head_dim), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(head_dim) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = enc(map, dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, const_cast<void*>(pool), dims, strides, box, elem_strides,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pkv::fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
  return PKV_OK;
}

// An INT8 code pool seen as a 2-D uint8 tensor of num_blocks*num_kv_heads*16
// rows by head_dim columns, read in boxes of 16 rows x min(head_dim, 128)
// bytes with the 128-byte swizzle (the 64-byte one for 64-byte rows).
pkv_status_t code_tensor_map(CUtensorMap* map, const void* pool, int64_t rows, int head_dim) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return pkv::fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cuuint64_t(head_dim), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(head_dim)};
  const cuuint32_t box[2] = {cuuint32_t(head_dim < 128 ? head_dim : 128), PKV_BLOCK_SIZE};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, box,
                         elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         head_dim < 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pkv::fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (uint8) failed (CUresult %d)", int(r));
  return PKV_OK;
}

pkv_status_t cuda_status(cudaError_t err, const char* what) {
  if (err == cudaSuccess) return pkv::ok();
  return pkv::fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

// Launches the prefix plan kernel into a shared-prefix workspace (its layout
// as prefix_layout gives it for these sizes).
pkv_status_t launch_prefix_plan_ws(const int32_t* context_lens, const int32_t* block_tables, int num_seqs,
                                   int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                                   char* ws, cudaStream_t stream) {
  const SplitLayout split = split_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, pkv::kPrefixMaxParts);
  const PrefixLayout pre = prefix_layout(split.total, num_seqs);
  int slots = 0;
  const pkv_status_t st = prefix_slots(head_dim, &slots);
  if (st != PKV_OK) return st;
  return cuda_status(pkv::launch_prefix_plan(context_lens, block_tables, num_seqs, max_blocks_per_seq, num_kv_heads,
                                             slots, prefix_max_members(num_q_heads, num_kv_heads),
                                             reinterpret_cast<int4*>(ws + pre.header_offset),
                                             reinterpret_cast<int4*>(ws + pre.groups_offset),
                                             reinterpret_cast<int4*>(ws + pre.chunks_offset),
                                             reinterpret_cast<int32_t*>(ws + pre.others_offset),
                                             reinterpret_cast<unsigned int*>(ws + split.counter_offset), stream),
                     "prefix plan");
}

bool supported_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

// Trace buffer of PKV_TRACE builds (pkv_set_trace_buffer), per process.
unsigned long long* g_trace_buffer = nullptr;
int g_trace_records = 0;

}  // namespace

extern "C" {

int pkv_trace_enabled(void) { return pkv::kTrace ? 1 : 0; }

pkv_status_t pkv_set_trace_buffer(unsigned long long* device_buffer, int records) {
  if (!pkv::kTrace) return pkv::fail(PKV_ERR_UNSUPPORTED, "this build records no traces (build with PKV_TRACE=1)");
  if (records < 0 || (records > 0 && !device_buffer) || !aligned(device_buffer, 8))
    return pkv::fail(PKV_ERR_INVALID_ARG, "set_trace_buffer: bad buffer");
  g_trace_buffer = records > 0 ? device_buffer : nullptr;
  g_trace_records = records;
  return pkv::ok();
}

pkv_status_t pkv_trace_stamp(unsigned long long* device_word, void* stream) {
  if (!device_word || !aligned(device_word, 8)) return pkv::fail(PKV_ERR_INVALID_ARG, "trace_stamp: bad word");
  return cuda_status(pkv::launch_trace_stamp(device_word, static_cast<cudaStream_t>(stream)), "trace_stamp launch");
}

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

int pkv_paged_attention_partition(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int max_blocks_per_seq, int partition_size) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  const int p = choose_partition(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, partition_size);
  Plan plan;
  if (plan_decode(max_blocks_per_seq, p, &plan) != PKV_OK) return 0;
  if (p == kBalanced) return kBalanced;
  if (p == kSharedPrefix)
    return prefix_fits(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq) ? kSharedPrefix : 0;
  return plan.max_parts <= 1 ? -1 : plan.part_tokens;
}

size_t pkv_paged_attention_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int max_blocks_per_seq,
                                          int partition_size) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  const int p = choose_partition(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, partition_size);
  Plan plan;
  if (plan_decode(max_blocks_per_seq, p, &plan) != PKV_OK) return 0;
  if (p == kBalanced) {
    if (num_q_heads % num_kv_heads != 0) return 0;
    return sk_layout(num_seqs, num_q_heads, num_kv_heads, head_dim).total;
  }
  if (p == kSharedPrefix) {
    if (!prefix_fits(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq)) return 0;
    return prefix_layout(split_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, pkv::kPrefixMaxParts).total,
                         num_seqs)
        .total;
  }
  return split_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, plan.max_parts).total +
         plan_bytes(num_seqs, num_kv_heads, plan.max_parts);
}

}  // extern "C"

namespace {

// Blocks a sliding window of `window` tokens can touch (it may start inside a
// block), capped by the table width; the whole table without a window.
int window_blocks(int max_blocks_per_seq, int window) {
  if (window <= 0) return max_blocks_per_seq;
  const int64_t wb = (int64_t(window) + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE + 1;
  return wb < max_blocks_per_seq ? int(wb) : max_blocks_per_seq;
}

pkv_status_t decode_impl(void* out, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                         int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                         int num_blocks, float scale, pkv_dtype_t dtype, int window, int partition_size,
                         void* workspace, size_t workspace_bytes, bool planned, pkv_stream_t stream) {
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

  // With a sliding window the partitions cover the window, not the table.
  const int plan_blocks = window_blocks(max_blocks_per_seq, window);
  const int p = choose_partition(num_seqs, num_q_heads, num_kv_heads, head_dim, plan_blocks, partition_size);
  Plan plan;
  pkv_status_t st = plan_decode(plan_blocks, p, &plan);
  if (st != PKV_OK) return st;
  const bool balanced = p == kBalanced;
  const bool shared_prefix = p == kSharedPrefix;
  if (shared_prefix && (window > 0 || !prefix_fits(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq)))
    return pkv::fail(PKV_ERR_UNSUPPORTED,
                     "the shared-prefix schedule takes 2..%d sequences, at most 4 query heads per KV head, tables "
                     "of at most %d blocks and no sliding window",
                     pkv::kOrderMaxSeqs, pkv::kPrefixMaxBlocks);
  if (balanced && window > 0)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "the balanced schedule takes no sliding window");
  if (balanced && !balanced_fits(num_seqs, num_q_heads, num_kv_heads, head_dim))
    return pkv::fail(PKV_ERR_UNSUPPORTED, "the balanced schedule takes at most %d sequences at these sizes",
                     pkv::decode_sk_max_seqs(head_dim, round_pow2_group(group)));
  const SplitLayout lay = split_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, plan.max_parts);
  const SkLayout sk = sk_layout(num_seqs, num_q_heads, num_kv_heads, head_dim);
  const size_t ord = (balanced || shared_prefix) ? 0 : plan_bytes(num_seqs, num_kv_heads, plan.max_parts);
  const SplitLayout pre_split = split_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, pkv::kPrefixMaxParts);
  const PrefixLayout pre = prefix_layout(pre_split.total, num_seqs);
  const size_t need = balanced ? sk.total : shared_prefix ? pre.total : lay.total + ord;
  if (int64_t(num_blocks) * num_kv_heads * PKV_BLOCK_SIZE > INT32_MAX)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * 16 exceeds 2^31 rows");
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
    return pkv::fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) required, got %zu at %p",
                     need, workspace_bytes, workspace);

  unsigned int* status = nullptr;
  st = status_word(&status);
  if (st != PKV_OK) return st;

  const int gpad = round_pow2_group(group);
  // boxes of 16, 8 and 4 rows (the tensor-core kernel copies partial last
  // tiles in 4-row multiples; the balanced schedule uses the first pair)
  alignas(64) CUtensorMap kmap[3], vmap[3];
  if (gpad >= 2 || shared_prefix) {
    const int64_t rows = int64_t(num_blocks) * num_kv_heads * PKV_BLOCK_SIZE;
    for (int i = 0; i < 3; ++i) {
      st = pool_tensor_map(&kmap[i], k_pool, rows, head_dim, dtype, PKV_BLOCK_SIZE >> i);
      if (st != PKV_OK) return st;
      st = pool_tensor_map(&vmap[i], v_pool, rows, head_dim, dtype, PKV_BLOCK_SIZE >> i);
      if (st != PKV_OK) return st;
    }
  }

  if (balanced) {
    pkv::SkArgs b;
    b.out = out;
    b.q = q;
    b.k_pool = k_pool;
    b.v_pool = v_pool;
    b.block_tables = block_tables;
    b.context_lens = context_lens;
    b.slots = static_cast<float*>(workspace);
    b.counters = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) + sk.counter_offset);
    b.status = status;
    b.num_seqs = num_seqs;
    b.num_q_heads = num_q_heads;
    b.num_kv_heads = num_kv_heads;
    b.group = group;
    b.max_blocks_per_seq = max_blocks_per_seq;
    b.num_blocks = num_blocks;
    b.slot_floats = sk.slot_floats;
    b.scale_log2 = scale * 1.4426950408889634f;
    // Arrival counters start at zero on every call; the slots need no initialisation.
    cudaError_t err = cudaMemsetAsync(b.counters, 0, sk.counter_bytes, stream);
    if (err != cudaSuccess) return cuda_status(err, "clear arrival counters");
    err = dtype == PKV_F16 ? pkv::launch_decode_sk_f16(b, head_dim, gpad, kmap, vmap, stream)
                           : pkv::launch_decode_sk_bf16(b, head_dim, gpad, kmap, vmap, stream);
    return cuda_status(err, "paged_attention_decode launch");
  }

  pkv::DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.part_o = lay.total > 0 ? static_cast<float*>(workspace) : nullptr;
  a.part_ml = lay.total > 0 ? reinterpret_cast<float2*>(static_cast<char*>(workspace) + lay.ml_offset) : nullptr;
  a.counters = lay.total > 0 ? reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) + lay.counter_offset)
                             : nullptr;
  // The launch plan: made here for batches of at least kOrderKernelMinSeqs
  // sequences, read as the caller made it for a planned call, else (smaller
  // batches) ranked in every CTA.
  int4* plan_hdr = ord > 0 ? reinterpret_cast<int4*>(static_cast<char*>(workspace) + lay.total) : nullptr;
  const bool make_plan = plan_hdr && !planned && num_seqs >= kOrderKernelMinSeqs;
  const bool use_plan = plan_hdr && (planned || make_plan);
  a.order = use_plan ? reinterpret_cast<const int32_t*>(plan_hdr + 1) : nullptr;
  a.plan = use_plan ? plan_hdr : nullptr;
  a.plan_rows = use_plan && round_pow2_group(group) >= 2 && window <= 0 ? plan_rows_of(plan_hdr, num_seqs) : nullptr;
  a.status = status;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.part_tokens = plan.part_tokens;
  a.max_parts = plan.max_parts;
  // Ranking the batch costs each CTA a dependent read of all lengths (about a
  // microsecond); it pays off only when the grid has few waves, where a long
  // sequence started last sets the end time (measured on GB300: -9 % on the
  // LLaMA-13B layer at 2560 CTAs, +7 % on the OPT-66B sampling batch at 9216).
  a.long_first = long_first_grid(num_seqs, num_kv_heads, plan.max_parts) ? 1 : 0;
  a.window = window > 0 ? window : 0;
  a.trace = g_trace_buffer;
  a.trace_records = g_trace_records;
  a.scale_log2 = scale * 1.4426950408889634f;

  cudaError_t err = cudaSuccess;
  if (shared_prefix) {
    // The prefix plan (made here, or by pkv_paged_attention_plan for a planned
    // call) groups siblings and zeroes the merge counters; a chunk's CTA reads
    // its group's shared prompt blocks once and each member's own blocks, the
    // other CTAs take the sequences outside any group.
    char* ws = static_cast<char*>(workspace);
    a.long_first = 0;
    a.order = nullptr;
    a.plan = nullptr;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_ml = reinterpret_cast<float2*>(ws + pre_split.ml_offset);
    a.counters = reinterpret_cast<unsigned int*>(ws + pre_split.counter_offset);
    a.prefix_header = reinterpret_cast<int4*>(ws + pre.header_offset);
    a.prefix_groups = reinterpret_cast<int4*>(ws + pre.groups_offset);
    a.prefix_chunks = reinterpret_cast<int4*>(ws + pre.chunks_offset);
    a.prefix_others = reinterpret_cast<int32_t*>(ws + pre.others_offset);
    a.prefix_slots = pre.max_chunks;
    if (!planned) {
      st = launch_prefix_plan_ws(context_lens, block_tables, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                 max_blocks_per_seq, ws, stream);
      if (st != PKV_OK) return st;
    }
    // one launch of the tensor-core kernel with rows of kPrefixRows query rows:
    // the chunk CTAs first, then the sequences outside any group
    err = dtype == PKV_F16 ? pkv::launch_decode_f16(a, head_dim, pkv::kPrefixRows, kmap, vmap, stream)
                           : pkv::launch_decode_bf16(a, head_dim, pkv::kPrefixRows, kmap, vmap, stream);
    return cuda_status(err, "paged_attention_decode launch");
  }
  if (lay.total > 0) {
    // The partition counters start at zero on every call; the partials need no initialisation.
    err = cudaMemsetAsync(a.counters, 0, lay.counter_bytes, stream);
    if (err != cudaSuccess) return cuda_status(err, "clear split-K counters");
  }
  if (make_plan) {
    err = pkv::launch_seq_order(context_lens, num_seqs, max_blocks_per_seq * PKV_BLOCK_SIZE, a.window, true, plan_hdr,
                                block_tables, max_blocks_per_seq, plan_rows_of(plan_hdr, num_seqs), stream);
    if (err != cudaSuccess) return cuda_status(err, "launch plan");
  }
  err = dtype == PKV_F16 ? pkv::launch_decode_f16(a, head_dim, gpad, kmap, vmap, stream)
                         : pkv::launch_decode_bf16(a, head_dim, gpad, kmap, vmap, stream);
  return cuda_status(err, "paged_attention_decode launch");
}

}  // namespace

extern "C" {

pkv_status_t pkv_paged_attention_decode(void* out, const void* q, const void* k_pool,
                                        const void* v_pool, const int32_t* block_tables,
                                        const int32_t* context_lens, int num_seqs,
                                        int num_q_heads, int num_kv_heads, int head_dim,
                                        int max_blocks_per_seq, int num_blocks, float scale,
                                        pkv_dtype_t dtype, int partition_size, void* workspace,
                                        size_t workspace_bytes, pkv_stream_t stream) {
  return decode_impl(out, q, k_pool, v_pool, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, max_blocks_per_seq, num_blocks, scale, dtype, 0, partition_size, workspace,
                     workspace_bytes, false, stream);
}

pkv_status_t pkv_paged_attention_decode_planned(void* out, const void* q, const void* k_pool, const void* v_pool,
                                                const int32_t* block_tables, const int32_t* context_lens,
                                                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                                int max_blocks_per_seq, int num_blocks, float scale,
                                                pkv_dtype_t dtype, int partition_size, void* workspace,
                                                size_t workspace_bytes, pkv_stream_t stream) {
  return decode_impl(out, q, k_pool, v_pool, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, max_blocks_per_seq, num_blocks, scale, dtype, 0, partition_size, workspace,
                     workspace_bytes, true, stream);
}

pkv_status_t pkv_paged_attention_plan(const int32_t* context_lens, const int32_t* block_tables, int num_seqs,
                                      int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                                      int partition_size, void* workspace, size_t workspace_bytes,
                                      pkv_stream_t stream) {
  if (num_seqs < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_seqs < 0");
  if (num_seqs == 0) return pkv::ok();
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                     num_q_heads, num_kv_heads);
  if (max_blocks_per_seq <= 0) return pkv::fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be > 0");
  if (!context_lens || !aligned(context_lens, 4))
    return pkv::fail(PKV_ERR_INVALID_ARG, "context_lens must be a 4-byte aligned pointer");
  const int p = choose_partition(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, partition_size);
  Plan plan;
  pkv_status_t st = plan_decode(max_blocks_per_seq, p, &plan);
  if (st != PKV_OK) return st;
  if (p == kBalanced) return pkv::ok();  // the balanced schedule takes no plan
  if (p == kSharedPrefix) {
    if (!prefix_fits(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq))
      return pkv::fail(PKV_ERR_UNSUPPORTED, "these sizes take no shared-prefix schedule");
    if (!block_tables || !aligned(block_tables, 4))
      return pkv::fail(PKV_ERR_INVALID_ARG, "the shared-prefix plan reads block_tables (4-byte aligned)");
    const PrefixLayout pre = prefix_layout(
        split_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, pkv::kPrefixMaxParts).total, num_seqs);
    if (!workspace || workspace_bytes < pre.total || !aligned(workspace, 16))
      return pkv::fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) required, got %zu at %p",
                       pre.total, workspace_bytes, workspace);
    return launch_prefix_plan_ws(context_lens, block_tables, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                 max_blocks_per_seq, static_cast<char*>(workspace), stream);
  }
  const SplitLayout lay = split_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, plan.max_parts);
  const size_t ord = plan_bytes(num_seqs, num_kv_heads, plan.max_parts);
  if (ord == 0) return pkv::ok();        // nothing to plan: natural order
  if (!workspace || workspace_bytes < lay.total + ord || !aligned(workspace, 16))
    return pkv::fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) required, got %zu at %p",
                     lay.total + ord, workspace_bytes, workspace);
  int4* plan_hdr = reinterpret_cast<int4*>(static_cast<char*>(workspace) + lay.total);
  return cuda_status(pkv::launch_seq_order(context_lens, num_seqs, max_blocks_per_seq * PKV_BLOCK_SIZE, 0,
                                           num_seqs >= kOrderKernelMinSeqs, plan_hdr, block_tables,
                                           max_blocks_per_seq, plan_rows_of(plan_hdr, num_seqs), stream),
                     "launch plan");
}

pkv_status_t pkv_paged_attention_decode_sliding(void* out, const void* q, const void* k_pool, const void* v_pool,
                                                const int32_t* block_tables, const int32_t* context_lens,
                                                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                                int max_blocks_per_seq, int num_blocks, float scale,
                                                pkv_dtype_t dtype, int sliding_window, int partition_size,
                                                void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  return decode_impl(out, q, k_pool, v_pool, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, max_blocks_per_seq, num_blocks, scale, dtype, sliding_window > 0 ? sliding_window : 0,
                     partition_size, workspace, workspace_bytes, false, stream);
}

size_t pkv_paged_attention_sliding_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                                  int max_blocks_per_seq, int sliding_window, int partition_size) {
  if (max_blocks_per_seq <= 0) return 0;
  if (sliding_window > 0 && (partition_size == kBalanced || partition_size == kSharedPrefix)) return 0;
  return pkv_paged_attention_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                            window_blocks(max_blocks_per_seq, sliding_window), partition_size);
}

namespace {

pkv_status_t decode_int8_impl(void* out, const void* q, const int8_t* k_cache, const int8_t* v_cache,
                              const float* k_scale, const float* v_scale, const int32_t* block_tables,
                              const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                              int head_dim, int max_blocks_per_seq, int num_blocks, float scale, pkv_dtype_t dtype,
                              int partition_size, void* workspace, size_t workspace_bytes, bool planned,
                              cudaStream_t stream) {
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
  if (!out || !q || !k_cache || !v_cache || !k_scale || !v_scale || !block_tables || !context_lens)
    return pkv::fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(k_scale, 16) || !aligned(v_scale, 16))
    return pkv::fail(PKV_ERR_INVALID_ARG, "out, q, caches and scales must be 16-byte aligned");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4))
    return pkv::fail(PKV_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");
  const int p = choose_partition(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, partition_size);
  if (p == kBalanced) return pkv::fail(PKV_ERR_UNSUPPORTED, "the INT8 cache has no balanced schedule");
  const bool shared_prefix = p == kSharedPrefix;
  if (shared_prefix && !prefix_fits(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq))
    return pkv::fail(PKV_ERR_UNSUPPORTED,
                     "the shared-prefix schedule takes 2..%d sequences, at most 4 query heads per KV head and "
                     "tables of at most %d blocks",
                     pkv::kOrderMaxSeqs, pkv::kPrefixMaxBlocks);
  if (shared_prefix && !pkv::decode_int8_uses_tensor_maps())
    return pkv::fail(PKV_ERR_UNSUPPORTED, "the shared-prefix schedule needs the tensor-core INT8 tile");
  Plan plan;
  pkv_status_t st = plan_decode(max_blocks_per_seq, p, &plan);
  if (st != PKV_OK) return st;
  if (int64_t(num_blocks) * num_kv_heads * PKV_BLOCK_SIZE > INT32_MAX)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * 16 exceeds 2^31 rows");
  const SplitLayout lay = split_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, plan.max_parts);
  const size_t ord = shared_prefix ? 0 : plan_bytes(num_seqs, num_kv_heads, plan.max_parts);
  const SplitLayout pre_split = split_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, pkv::kPrefixMaxParts);
  const PrefixLayout pre = prefix_layout(pre_split.total, num_seqs);
  const size_t need = shared_prefix ? pre.total : lay.total + ord;
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
    return pkv::fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) required, got %zu at %p",
                     need, workspace_bytes, workspace);
  unsigned int* status = nullptr;
  st = status_word(&status);
  if (st != PKV_OK) return st;

  pkv::DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_pool = k_cache;
  a.v_pool = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.part_o = lay.total > 0 ? static_cast<float*>(workspace) : nullptr;
  a.part_ml = lay.total > 0 ? reinterpret_cast<float2*>(static_cast<char*>(workspace) + lay.ml_offset) : nullptr;
  a.counters = lay.total > 0 ? reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) + lay.counter_offset)
                             : nullptr;
  // The launch plan, as for the 16-bit cache: made here for batches of at
  // least kOrderKernelMinSeqs sequences, read as the caller made it for a
  // planned call, else ranked in every CTA.
  int4* plan_hdr = ord > 0 ? reinterpret_cast<int4*>(static_cast<char*>(workspace) + lay.total) : nullptr;
  const bool make_plan = plan_hdr && !planned && num_seqs >= kOrderKernelMinSeqs;
  const bool use_plan = plan_hdr && (planned || make_plan);
  a.order = use_plan ? reinterpret_cast<const int32_t*>(plan_hdr + 1) : nullptr;
  a.plan = use_plan ? plan_hdr : nullptr;
  a.status = status;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.part_tokens = plan.part_tokens;
  a.max_parts = plan.max_parts;
  a.long_first = long_first_grid(num_seqs, num_kv_heads, plan.max_parts) ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  alignas(64) CUtensorMap kmap, vmap;
  if (pkv::decode_int8_uses_tensor_maps()) {
    const int64_t rows = int64_t(num_blocks) * num_kv_heads * PKV_BLOCK_SIZE;
    st = code_tensor_map(&kmap, k_cache, rows, head_dim);
    if (st != PKV_OK) return st;
    st = code_tensor_map(&vmap, v_cache, rows, head_dim);
    if (st != PKV_OK) return st;
  }
  cudaError_t err = cudaSuccess;
  int gpad = round_pow2_group(group);
  if (shared_prefix) {
    // The prefix plan (made here, or by pkv_paged_attention_plan for a planned
    // call; its layout does not depend on the cache's element type).
    char* ws = static_cast<char*>(workspace);
    a.long_first = 0;
    a.order = nullptr;
    a.plan = nullptr;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_ml = reinterpret_cast<float2*>(ws + pre_split.ml_offset);
    a.counters = reinterpret_cast<unsigned int*>(ws + pre_split.counter_offset);
    a.prefix_header = reinterpret_cast<int4*>(ws + pre.header_offset);
    a.prefix_groups = reinterpret_cast<int4*>(ws + pre.groups_offset);
    a.prefix_chunks = reinterpret_cast<int4*>(ws + pre.chunks_offset);
    a.prefix_others = reinterpret_cast<int32_t*>(ws + pre.others_offset);
    a.prefix_slots = pre.max_chunks;
    if (!planned) {
      st = launch_prefix_plan_ws(context_lens, block_tables, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                 max_blocks_per_seq, ws, stream);
      if (st != PKV_OK) return st;
    }
    gpad = pkv::kPrefixRows;
  } else {
    if (lay.total > 0) {
      err = cudaMemsetAsync(a.counters, 0, lay.counter_bytes, stream);
      if (err != cudaSuccess) return cuda_status(err, "clear split-K counters");
    }
    if (make_plan) {
      err = pkv::launch_seq_order(context_lens, num_seqs, max_blocks_per_seq * PKV_BLOCK_SIZE, 0, true, plan_hdr,
                                  block_tables, max_blocks_per_seq, plan_rows_of(plan_hdr, num_seqs), stream);
      if (err != cudaSuccess) return cuda_status(err, "launch plan");
    }
  }
  err = pkv::launch_decode_int8(a, dtype == PKV_BF16, head_dim, gpad, &kmap, &vmap, stream);
  return cuda_status(err, "paged_attention_decode_int8 launch");
}

}  // namespace

pkv_status_t pkv_paged_attention_decode_int8(void* out, const void* q, const int8_t* k_cache,
                                             const int8_t* v_cache, const float* k_scale, const float* v_scale,
                                             const int32_t* block_tables, const int32_t* context_lens,
                                             int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                             int max_blocks_per_seq, int num_blocks, float scale,
                                             pkv_dtype_t dtype, int partition_size, void* workspace,
                                             size_t workspace_bytes, pkv_stream_t stream) {
  return decode_int8_impl(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, num_seqs,
                          num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype,
                          partition_size, workspace, workspace_bytes, false, static_cast<cudaStream_t>(stream));
}

pkv_status_t pkv_paged_attention_decode_int8_planned(void* out, const void* q, const int8_t* k_cache,
                                                     const int8_t* v_cache, const float* k_scale,
                                                     const float* v_scale, const int32_t* block_tables,
                                                     const int32_t* context_lens, int num_seqs, int num_q_heads,
                                                     int num_kv_heads, int head_dim, int max_blocks_per_seq,
                                                     int num_blocks, float scale, pkv_dtype_t dtype,
                                                     int partition_size, void* workspace, size_t workspace_bytes,
                                                     pkv_stream_t stream) {
  return decode_int8_impl(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, num_seqs,
                          num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, num_blocks, scale, dtype,
                          partition_size, workspace, workspace_bytes, true, static_cast<cudaStream_t>(stream));
}

pkv_status_t pkv_reshape_and_cache_int8(const void* k, const void* v, pkv_dtype_t dtype, int8_t* k_cache,
                                        int8_t* v_cache, float* k_scale, float* v_scale,
                                        const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                        int head_dim, int num_blocks, pkv_stream_t stream) {
  if (num_tokens < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0) return pkv::ok();
  if (num_kv_heads <= 0 || num_blocks <= 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be > 0");
  if (!supported_head_dim(head_dim)) return pkv::fail(PKV_ERR_UNSUPPORTED, "head_dim %d (64, 128 or 256)", head_dim);
  if (dtype != PKV_F16 && dtype != PKV_BF16) return pkv::fail(PKV_ERR_UNSUPPORTED, "dtype %d", int(dtype));
  if (!k || !v || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
    return pkv::fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(k_scale, 16) || !aligned(v_scale, 16) || !aligned(slot_mapping, 8))
    return pkv::fail(PKV_ERR_INVALID_ARG, "k, v, caches and scales must be 16-byte aligned, slot_mapping 8-byte aligned");
  if (int64_t(num_tokens) * num_kv_heads > int64_t(UINT32_MAX) * 8)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "too many tokens for one launch");
  unsigned int* status = nullptr;
  pkv_status_t st = status_word(&status);
  if (st != PKV_OK) return st;
  return cuda_status(pkv::launch_reshape_and_cache_int8(k, v, dtype == PKV_BF16, k_cache, v_cache, k_scale, v_scale,
                                                        slot_mapping, num_tokens, num_kv_heads, head_dim,
                                                        num_blocks, status, stream),
                     "reshape_and_cache_int8 launch");
}

pkv_status_t pkv_copy_blocks_int8(int8_t* k_cache, int8_t* v_cache, float* k_scale, float* v_scale,
                                  const int64_t* src_dst_pairs, int num_pairs, int num_kv_heads, int head_dim,
                                  int num_blocks, pkv_stream_t stream) {
  if (num_pairs < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_pairs < 0");
  if (num_pairs == 0) return pkv::ok();
  if (num_pairs > 65535) return pkv::fail(PKV_ERR_UNSUPPORTED, "num_pairs %d > 65535", num_pairs);
  if (num_kv_heads <= 0 || num_blocks <= 0) return pkv::fail(PKV_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be > 0");
  if (!supported_head_dim(head_dim)) return pkv::fail(PKV_ERR_UNSUPPORTED, "head_dim %d (64, 128 or 256)", head_dim);
  if (!k_cache || !v_cache || !k_scale || !v_scale || !src_dst_pairs) return pkv::fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_scale, 16) || !aligned(v_scale, 16) ||
      !aligned(src_dst_pairs, 8))
    return pkv::fail(PKV_ERR_INVALID_ARG, "caches and scales must be 16-byte aligned, pairs 8-byte aligned");
  unsigned int* status = nullptr;
  pkv_status_t st = status_word(&status);
  if (st != PKV_OK) return st;
  cudaError_t err = pkv::launch_copy_blocks_bytes(k_cache, v_cache, src_dst_pairs, num_pairs,
                                                  int64_t(num_kv_heads) * PKV_BLOCK_SIZE * head_dim, num_blocks,
                                                  status, stream);
  if (err != cudaSuccess) return cuda_status(err, "copy_blocks_int8 launch (codes)");
  return cuda_status(pkv::launch_copy_blocks_bytes(k_scale, v_scale, src_dst_pairs, num_pairs,
                                                   int64_t(num_kv_heads) * PKV_BLOCK_SIZE * 4, num_blocks, status,
                                                   stream),
                     "copy_blocks_int8 launch (scales)");
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

pkv_status_t pkv_selftest_bounded_wait(uint32_t limit_us, pkv_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000)
    return pkv::fail(PKV_ERR_INVALID_ARG, "selftest_bounded_wait: limit_us must be in 1..1000000");
  unsigned int* status = nullptr;
  pkv_status_t st = status_word(&status);
  if (st != PKV_OK) return st;
  return cuda_status(pkv::launch_bounded_wait_selftest(1000ull * limit_us, status, stream),
                     "bounded-wait self-test launch");
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
