/*
 * paged_kv.h -- C ABI of the PagedAttention decode library (GB300, sm_103a).
 *
 * The library implements the decode-time hot path of PagedAttention: each
 * running sequence's new query token attends over that sequence's KV cache,
 * which is stored as fixed 16-token physical blocks scattered through a shared
 * pool and reached through a per-sequence block table; next to it sit the
 * write of each step's new K/V into its slot, the copy-on-write block copy,
 * and a host-side block manager that produces the tables and slot maps.
 *
 * Sources (web pages on PagedAttention, by title and section):
 *  [G]  "PagedAttention（ページドアテンション）" glossary entry (jisaku.com):
 *       "PagedAttentionの解決策" (16-token blocks, block table logical ->
 *       physical, blocks need not be contiguous), "コピーオンライト
 *       （Copy-on-Write）共有" (parallel sampling shares prompt blocks),
 *       "他のKVキャッシュ最適化との組み合わせ" (GQA + paging).
 *  [B]  "数万トークンでもVRAMが溢れない！LLM推論を爆速化する「PagedAttention」の全貌"
 *       (blog): "OSの知恵をGPUへ" (on-demand blocks, waste only in the last
 *       block, sharing by reference count).
 *  [S]  abeam.tech summary of "Efficient Memory Management for Large Language
 *       Model Serving with PagedAttention": "用語解説" (block table,
 *       Copy-on-Write), "技術の仕組み" (the kernel reads KV through the block
 *       table), "KV キャッシュマネージャ" (fill the last block, allocate when
 *       full, return blocks on finish), "並列サンプリングやビームサーチでの共有"
 *       (copy only when a write reaches a shared block), "よくある質問" (not a
 *       new attention formula).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Block size is 16 tokens ([G], [B]); it is fixed at compile time.
 *  - Element type T is IEEE fp16 or bfloat16 (pkv_dtype_t) for q, out, K, V.
 *  - Layouts (all row-major, densely packed, element strides implied):
 *      q, out        : T[num_seqs][num_q_heads][head_dim]
 *      k_pool, v_pool: T[num_blocks][num_kv_heads][16][head_dim]
 *                      (one (block, kv head) tile is a contiguous 16*head_dim
 *                      span, 4 KiB at head_dim 128)
 *      block_tables  : int32[num_seqs][max_blocks_per_seq]; entries past
 *                      ceil(context_len/16) are never read (pad with -1)
 *      context_lens  : int32[num_seqs]; 0 marks an empty (padding) sequence
 *      slot_mapping  : int64[num_tokens]; slot = block * 16 + offset, < 0 skips
 *      src_dst_pairs : int64[num_pairs][2]
 *    Token position p of sequence s lives in block block_tables[s][p / 16],
 *    slot p % 16 ([G], "PagedAttentionの解決策").
 *  - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  - Device pointers are owned by the caller; the library never allocates
 *    device memory. Scratch for split-K decode comes from a caller-provided
 *    workspace (pkv_paged_attention_workspace_size).
 *  - Every GPU call is asynchronous on `stream` (a cudaStream_t; NULL means
 *    the legacy default stream) and returns after the launch. Scalar
 *    arguments are checked on the host before anything is launched; on a
 *    failed check nothing is launched and the status says why
 *    (pkv_last_error_string gives the detail, per calling thread).
 *  - Per-device state of the library (the device status word, the scratch of
 *    pkv_paged_attention_decode_noalloc) is looked up on the current CUDA
 *    device, once per device index, and kept for the life of the process:
 *    make the device of the pointers and of `stream` current before a call,
 *    and do not use the library across a cudaDeviceReset.
 *  - Device-resident indices (block ids, context lengths, slots, pairs) are
 *    checked by the kernels. A bad index never faults: the kernel records a
 *    flag in the device status word (pkv_device_status), skips the access or
 *    clamps it into range, and the affected output is unspecified.
 *  - pointers must be 16-byte aligned (q, out, pools, k, v) and 4/8-byte
 *    aligned for the int32/int64 arrays.
 */
#ifndef PAGED_KV_H_
#define PAGED_KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_BLOCK_SIZE 16

/* Status of every call. */
typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* a size, pointer or index argument is out of range */
  PKV_ERR_UNSUPPORTED = 2,   /* valid, but not built: dtype / head_dim / group size */
  PKV_ERR_OUT_OF_BLOCKS = 3, /* block manager: free list cannot satisfy the call */
  PKV_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, copy, attribute) */
  PKV_ERR_WORKSPACE = 5      /* workspace missing or smaller than required */
} pkv_status_t;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1 } pkv_dtype_t;

/* Flags of the device status word (pkv_device_status). */
#define PKV_DEV_BAD_BLOCK_ID    0x1u  /* block table entry outside [0, num_blocks) */
#define PKV_DEV_BAD_CONTEXT_LEN 0x2u  /* context_len < 0 or > max_blocks_per_seq*16 */
#define PKV_DEV_BAD_SLOT        0x4u  /* slot_mapping entry >= num_blocks*16 */
#define PKV_DEV_BAD_PAIR        0x8u  /* copy pair with src or dst outside the pool */
#define PKV_DEV_WAIT_TIMEOUT    0x10u /* a bounded wait on a copy gave up */
#define PKV_DEV_BAD_PLAN        0x20u /* a planned decode found no plan of its batch size */

typedef struct CUstream_st* pkv_stream_t; /* same type as cudaStream_t */

/* Library version string, static storage. */
const char* pkv_version(void);

/* Detail of the last failing call made by this thread ("" if none). */
const char* pkv_last_error_string(void);

/*
 * Reads the device status word of the current CUDA device into *flags_out
 * (PKV_DEV_* bits, 0 = no device-side check tripped since the last clear),
 * and clears it when `clear` is non-zero. Synchronises the device.
 */
pkv_status_t pkv_device_status(uint32_t* flags_out, int clear);

/*
 * Self-test of the kernels' bounded waits (no counterpart on the pages; a
 * failure-detection check). Launches one warp on `stream` that waits on a
 * shared-memory mbarrier for 16 bytes that no copy delivers, using the same
 * bounded wait as the decode kernels but with a limit of `limit_us`
 * microseconds (1..1000000). The wait runs out, the warp sets
 * PKV_DEV_WAIT_TIMEOUT in the device status word and exits; the context stays
 * usable. Read the flag with pkv_device_status.
 */
pkv_status_t pkv_selftest_bounded_wait(uint32_t limit_us, pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Decode attention                                                          */
/* ------------------------------------------------------------------------ */

/*
 * PagedAttention decode ([S] "技術の仕組み": the kernel follows the block
 * table to reach each sequence's non-contiguous KV; [S] "よくある質問": the
 * result is ordinary attention).
 *
 * For every sequence s and query head h (g = h / (num_q_heads/num_kv_heads),
 * L = context_lens[s]):
 *     out[s][h] = softmax_p( scale * <q[s][h], K_s[p]> ) . V_s[p],  p < L
 * with K_s[p] = k_pool[block_tables[s][p/16]][g][p%16] (V likewise).
 * Softmax, dot products and the weighted sum run in fp32 (online maximum and
 * running sum); out is rounded once to T. L == 0 writes zeros.
 *
 * partition_size (tokens) picks the schedule:
 *   0   library choice: one CTA per (sequence, KV head) when there are at
 *       least 608 such pairs (4 per SM), else split-K partitions just large
 *       enough to reach that many CTAs (>= 256 tokens);
 *  -1   one CTA per (sequence, KV head), no split;
 *  -2   balanced persistent schedule: every warp streams an equal share of
 *       the batch's 16-token tiles; items split between warps are merged by
 *       log-sum-exp (for heavily skewed length mixes; batches of up to 2048
 *       sequences at head_dim 128);
 *  -5   shared-prefix schedule, for parallel sampling and beam search
 *       ([S] "並列サンプリングやビームサーチでの共有": siblings' tables hold
 *       the same physical blocks for their common prompt): a one-CTA plan
 *       kernel groups consecutive sequences whose tables start with the same
 *       >= 4 physical blocks (at most 8 query rows a group: 8 / (query heads
 *       per KV head) members); one CTA per (group, KV head) copies each
 *       shared K/V tile once, multiplies it with every member's queries on
 *       the tensor cores, then streams each member's own blocks for that
 *       member's rows only. When the grid would be under one wave of
 *       resident CTAs, a group's blocks are split over up to 4 CTAs whose
 *       partials the last to finish merges by log-sum-exp. Sequences outside
 *       any group take one CTA each. Takes 2..1024 sequences, at most 4 query
 *       heads per KV head, tables of at most 256 blocks; groups form only
 *       from equal leading table entries, so a batch without sharing is
 *       still computed exactly. Siblings of one group with equal lengths and
 *       contents get bit-identical outputs;
 *  N>0  (multiple of 16) split-K partitions of N tokens, one CTA each, whose
 *       partial (max, sum, weighted V) are merged by log-sum-exp.
 * The result does not depend on the schedule beyond fp32 rounding.
 *
 * Supported: T in {fp16, bf16}; head_dim in {64, 128, 256};
 * num_q_heads % num_kv_heads == 0 with group size <= 8.
 *
 * workspace: device memory of at least
 * pkv_paged_attention_workspace_size(...) bytes for the same arguments, or
 * NULL when that size is 0. It holds fp32 partial results and one arrival
 * counter per (sequence, KV head): the last part of a split item to finish
 * merges the partials. The library clears the counters on `stream` before
 * each launch that uses them, so the workspace needs no initialisation and
 * may be reused by calls of any shape; calls that use one workspace must not
 * overlap on the GPU.
 *
 * Launch order: grids of at most 4096 CTAs start the sequences of at least
 * twice the batch's mean length (in 16-token tiles) first. For batches of 128
 * to 1024 sequences that order is computed once, by a one-CTA kernel launched
 * on `stream` ahead of the decode, into the plan region at the end of the
 * workspace (see pkv_paged_attention_plan); it also puts sequences of at most
 * 5/8 of the mean length last (each group in natural order). Smaller batches
 * are ranked in every CTA. The order changes only when the work starts,
 * never the results. The plan also holds, per grid row, the sequence, its
 * length and its first six block ids: the tensor-core kernel (groups of 2..8)
 * starts its first tile copies from them before its own reads of the length
 * and the table return, then compares them and copies again from the
 * sequence's own values if they differ.
 * That kernel reads context_lens and block_tables without waiting for the
 * previous kernel on the stream to finish when that kernel allows
 * programmatic early launch (the library's cache writes do, and touch
 * neither): a kernel that writes context_lens or block_tables and allows
 * early launch must not directly precede this call.
 *
 * Group size 1 runs on the CUDA cores; groups of 2..8 query heads per KV head
 * run the QK and PV products of each 16-token tile on the tensor cores (fp32
 * accumulation; the softmax weights enter as two 16-bit terms, keeping about
 * 16 significant bits).
 */
pkv_status_t pkv_paged_attention_decode(
    void* out, const void* q, const void* k_pool, const void* v_pool,
    const int32_t* block_tables, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int num_blocks, float scale, pkv_dtype_t dtype,
    int partition_size, void* workspace, size_t workspace_bytes,
    pkv_stream_t stream);

/* Bytes of workspace pkv_paged_attention_decode (and _decode_planned) needs
 * for these sizes: the split-K partials and counters, then the launch plan
 * (a 16-byte header, int32[num_seqs] rounded up to 16 bytes, then int4[2 *
 * num_seqs] of rows {sequence, length, block ids 0..5}) of batches of 2 to
 * 1024 sequences in grids of at most 4096 CTAs (see above); 0 for calls
 * without either. For
 * the shared-prefix schedule (-5): the split-K layout with 4 partitions (the
 * partials of split groups and one arrival counter per (sequence, KV head)),
 * then its plan: a 16-byte header, int4 groups[num_seqs / 2], int4
 * chunks[num_seqs] and int32[num_seqs] rounded up to 16 bytes.
 * Returns 0 for invalid sizes (and sizes -5 does not take) as well. */
size_t pkv_paged_attention_workspace_size(
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int partition_size);

/*
 * Launch plan of a decode step (the pages have no counterpart; a scheduling
 * convenience of this library). The order in which the decode grid takes the
 * sequences depends only on the batch (lengths and sizes), which every layer
 * of a decode step shares: this call computes it once -- the long-first order
 * described under pkv_paged_attention_decode (with the shortest sequences
 * last for batches of 128 or more), behind a 16-byte header -- into the plan
 * region of `workspace` (the bytes after the split-K scratch, see
 * pkv_paged_attention_workspace_size), and pkv_paged_attention_decode_planned
 * then uses it in every layer instead of ranking the batch itself.
 * Arguments as for pkv_paged_attention_decode; context_lens and block_tables
 * are read on `stream` (device memory, the same values the decode calls will
 * see). block_tables may be NULL except for the shared-prefix schedule: the
 * plan's rows then name no sequence and the decode reads every length and
 * block id itself. Does
 * nothing when the sizes need no plan (one sequence, more than 1024, grids of
 * more than 4096 CTAs, the balanced schedule). For the shared-prefix schedule
 * (partition_size -5) the plan holds the sibling groups instead; its decode
 * calls must see the same lengths and tables.
 */
pkv_status_t pkv_paged_attention_plan(const int32_t* context_lens, const int32_t* block_tables,
                                      int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                      int max_blocks_per_seq, int partition_size, void* workspace,
                                      size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_paged_attention_decode with the launch plan that pkv_paged_attention_plan
 * left in `workspace` for the same sizes: one kernel, no ranking. Same
 * arguments, semantics and results as pkv_paged_attention_decode (the plan
 * decides only when each sequence starts, never a result). A plan made from
 * other lengths or tables of a batch of the same size is still correct (the
 * start order is off, and first tile copies made from the plan's rows are
 * made again from the sequence's own length and ids). If the workspace holds no plan of this batch size, the
 * kernels flag PKV_DEV_BAD_PLAN and take the sequences in natural order,
 * still computing every output. The plan region must not be overwritten
 * between the plan and the decode calls that use it (a call with other sizes
 * on the same workspace can overwrite it).
 */
pkv_status_t pkv_paged_attention_decode_planned(
    void* out, const void* q, const void* k_pool, const void* v_pool,
    const int32_t* block_tables, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int num_blocks, float scale, pkv_dtype_t dtype,
    int partition_size, void* workspace, size_t workspace_bytes,
    pkv_stream_t stream);

/* The schedule a call with these sizes runs: -2 for the balanced persistent
 * schedule, -5 for the shared-prefix schedule, -1 for one CTA per (sequence,
 * KV head), else the split-K partition in tokens; 0 for invalid sizes (and
 * for -2 or -5 where those schedules do not take the sizes). Resolves
 * partition_size == 0 (never to -2 or -5). */
int pkv_paged_attention_partition(
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int partition_size);

/*
 * Decode attention that allocates nothing (the pages have no counterpart;
 * this is a deployment convenience of this library).
 *
 * Same arguments, semantics and results as pkv_paged_attention_decode,
 * without the workspace. For callers that cannot allocate device memory when
 * they decode -- e.g. a serving engine that reserves nearly all HBM for its
 * KV-cache pool, or host code that must not call cudaMalloc/cudaFree on its
 * critical path because they can synchronise the device -- split-K scratch
 * comes from a fixed array in the library's module memory of
 * PKV_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds
 * until the process exits. Sizes whose split-K scratch
 * (pkv_paged_attention_workspace_size) exceeds it return PKV_ERR_UNSUPPORTED
 * and launch nothing; a larger partition_size or -1 (one pass) needs less.
 *
 * The array used is the one of the current CUDA device, which must be the
 * device of `stream` and of every pointer argument. The first call on a
 * device looks up the array's device address (once per device index, with
 * that device current) and caches it for the life of the process; make that
 * first call before any stream capture. The cached address belongs to the
 * device's primary context: do not call this entry point again after a
 * cudaDeviceReset (or any other teardown of that context) in the same
 * process. Every call on a device shares the one array, which keeps the last
 * call's contents; the parts that must start at zero (the arrival counters of
 * the split-K, balanced and shared-prefix schedules) are cleared on `stream`
 * by every call (the last by its prefix plan kernel),
 * and everything else a call reads from the array it first writes itself.
 * Calls that overlap on the GPU (different streams, or different host
 * threads) race on it. No cudaMalloc, cudaFree or other allocating routine
 * is called.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */

pkv_status_t pkv_paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_pool, const void* v_pool,
    const int32_t* block_tables, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int num_blocks, float scale, pkv_dtype_t dtype,
    int partition_size, pkv_stream_t stream);

/*
 * Sliding-window decode ([G] "他のKVキャッシュ最適化との組み合わせ" names
 * sliding-window attention as a companion of paging; the page gives no
 * formula, so this library takes the usual one): the query of sequence s
 * attends over its last sliding_window tokens only,
 *   positions [max(0, L - W), L),  W = sliding_window,
 * and otherwise computes exactly what pkv_paged_attention_decode computes.
 * Block-table entries of blocks wholly before that range are never read (the
 * block manager may have released them, see pkv_bm_release_before).
 * sliding_window <= 0 means no window. partition_size as for
 * pkv_paged_attention_decode except -2 (balanced) and -5 (shared prefix),
 * which return PKV_ERR_UNSUPPORTED with a window; the split covers the
 * window, not the whole length.
 * The workspace must hold pkv_paged_attention_sliding_workspace_size bytes.
 */
pkv_status_t pkv_paged_attention_decode_sliding(
    void* out, const void* q, const void* k_pool, const void* v_pool,
    const int32_t* block_tables, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int num_blocks, float scale, pkv_dtype_t dtype,
    int sliding_window, int partition_size, void* workspace,
    size_t workspace_bytes, pkv_stream_t stream);

size_t pkv_paged_attention_sliding_workspace_size(int num_seqs, int num_q_heads,
                                                  int num_kv_heads, int head_dim,
                                                  int max_blocks_per_seq,
                                                  int sliding_window,
                                                  int partition_size);

/*
 * Diagnostics (the pages have no counterpart). Libraries built with
 * -DPKV_TRACE=1 (python -m paged_kv_cache_217_gb300.build --define
 * PKV_TRACE=1 --out-dir DIR) let each CTA of the one-pass and split decode
 * grids record eight 64-bit words into a device buffer of the caller's:
 * %globaltimer (ns) at its start, when its sequence is known, when its
 * length and block ids are known, when warp 0's first tile has landed, when
 * warp 0's tile loop ends and at its end; its SM; and its sequence (low 32
 * bits) and tile count (high 32 bits). Record i belongs to the CTA of linear
 * index i (blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
 * CTAs past `records` and CTAs of empty sequences write nothing. The buffer
 * applies to the decode calls that follow on any thread (NULL / 0 stops);
 * pkv_set_trace_buffer returns PKV_ERR_UNSUPPORTED in other builds, and
 * pkv_trace_enabled tells which build is loaded (1 or 0).
 */
int pkv_trace_enabled(void);
pkv_status_t pkv_set_trace_buffer(unsigned long long* device_buffer, int records);
/*
 * pkv_trace_stamp (every build) enqueues on `stream` a one-thread kernel that
 * writes %globaltimer (ns, the clock of the trace records) to the device word
 * `device_word` (8-byte aligned, caller-owned) when the stream reaches it:
 * stamps before and after a decode call place the call's CTAs within it.
 * The stamp is itself a launch, so the interval up to a stamp includes that
 * launch's latency. PKV_ERR_INVALID_ARG for a NULL or misaligned word.
 */
pkv_status_t pkv_trace_stamp(unsigned long long* device_word, void* stream);
/*
 * pkv_trace_empty_grid (every build) enqueues on `stream` a kernel of `ctas`
 * CTAs of `threads` threads with `smem_bytes` of dynamic shared memory that
 * reads and writes nothing, launched as the decode kernels are (programmatic
 * stream serialization). Timed between two events it gives the fixed cost of
 * a launch of that shape (dispatch of its CTAs and the kernel's completion),
 * which a decode call of the same grid pays before and after its own work.
 * PKV_ERR_INVALID_ARG unless ctas >= 1, 1 <= threads <= 1024 and
 * 0 <= smem_bytes <= 227 KB; a launch error is returned as PKV_ERR_CUDA.
 */
pkv_status_t pkv_trace_empty_grid(int ctas, int threads, int smem_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Cache writes and copy-on-write                                            */
/* ------------------------------------------------------------------------ */

/*
 * Writes each new token's K and V into its slot ([S] "KV キャッシュマネージャ":
 * tokens fill the last block of their sequence).
 *   k, v: T[num_tokens][num_kv_heads][head_dim]
 *   for t with slot = slot_mapping[t] >= 0 and every KV head g:
 *     k_pool[slot/16][g][slot%16][:] = k[t][g][:]   (v likewise)
 * A pure bit copy. Slots >= num_blocks*16 are skipped and flagged
 * (PKV_DEV_BAD_SLOT). Two tokens with the same slot race (unspecified winner).
 */
pkv_status_t pkv_reshape_and_cache(
    const void* k, const void* v, void* k_pool, void* v_pool,
    const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
    int head_dim, int num_blocks, pkv_dtype_t dtype, pkv_stream_t stream);

/*
 * Copy-on-write block copies ([S] "並列サンプリングやビームサーチでの共有",
 * [G] "コピーオンライト（Copy-on-Write）共有"): for each (src, dst) pair,
 * block src of both pools (all KV heads, all 16 slots) is copied to block dst.
 * src_dst_pairs is device memory. The pairs must not conflict: dst values
 * are distinct and no dst is also a src (pkv_check_copy_pairs tests this on
 * the host; the block manager's pairs satisfy it by construction). Pairs
 * with an id outside [0, num_blocks) are skipped and flagged.
 */
pkv_status_t pkv_copy_blocks(
    void* k_pool, void* v_pool, const int64_t* src_dst_pairs, int num_pairs,
    int num_kv_heads, int head_dim, int num_blocks, pkv_dtype_t dtype,
    pkv_stream_t stream);

/* Host check of a pair list (host memory): ids in range, dst distinct, no dst
 * used as a src. PKV_OK or PKV_ERR_INVALID_ARG. */
pkv_status_t pkv_check_copy_pairs(const int64_t* src_dst_pairs_host, int num_pairs,
                                  int num_blocks);

/* ------------------------------------------------------------------------ */
/* INT8 KV cache ([G] "他のKVキャッシュ最適化との組み合わせ": INT8             */
/* quantisation of the KV cache combines with paging, halving each block)    */
/* ------------------------------------------------------------------------ */
/*
 * The page names INT8 KV quantisation but gives no scheme; this library
 * takes the symmetric per-row reading: every stored row (block, KV head,
 * slot) of K and of V holds int8 codes and one fp32 scale,
 *   s = max_i |x_i| / 127,  c_i = rint(x_i / s)  (ties to even),
 * both computed in IEEE fp32 from the fp32 value of the 16-bit input, so
 * x_i ~= c_i * s with |x_i - c_i * s| <= s / 2. A row of zeros has s = 0 and
 * codes 0. Layouts:
 *   k_cache, v_cache : int8[num_blocks][num_kv_heads][16][head_dim]
 *   k_scale, v_scale : fp32[num_blocks][num_kv_heads][16]
 * head_dim is 64, 128 or 256. All four arrays must be 16-byte aligned.
 */

/*
 * Quantising cache write: for each t with slot = slot_mapping[t] >= 0 and
 * every KV head g, row k[t][g][:] (T = dtype) is quantised as above into
 * k_cache[slot/16][g][slot%16][:] and k_scale[slot/16][g][slot%16] (v
 * likewise). Slots >= num_blocks*16 are skipped and flagged
 * (PKV_DEV_BAD_SLOT). Codes and scales are bit-exact to the definition.
 */
pkv_status_t pkv_reshape_and_cache_int8(
    const void* k, const void* v, pkv_dtype_t dtype, int8_t* k_cache,
    int8_t* v_cache, float* k_scale, float* v_scale, const int64_t* slot_mapping,
    int num_tokens, int num_kv_heads, int head_dim, int num_blocks,
    pkv_stream_t stream);

/*
 * Decode over the INT8 cache: pkv_paged_attention_decode with every K row
 * read as c_K * s_K and every V row as c_V * s_V. q and out are T = dtype.
 * Same block tables, lengths, GQA rule, partition_size values (except -2,
 * the balanced schedule, which returns PKV_ERR_UNSUPPORTED; -5, the
 * shared-prefix schedule, runs as described there), workspace
 * (pkv_paged_attention_workspace_size with the same arguments) and error
 * behaviour. Internally the scores are q . c_K scaled by s_K (with one query
 * head per KV head and head_dim <= 128, q enters as two int8 digit planes,
 * q ~ s1 d1 + s2 d2, within max|q| / 64516 of q, so that the products run as
 * exact integer dot products), and s_V is folded into each softmax weight
 * (with a power of two per warp that keeps the weights inside the fp16
 * range).
 */
pkv_status_t pkv_paged_attention_decode_int8(
    void* out, const void* q, const int8_t* k_cache, const int8_t* v_cache,
    const float* k_scale, const float* v_scale, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
    int head_dim, int max_blocks_per_seq, int num_blocks, float scale,
    pkv_dtype_t dtype, int partition_size, void* workspace,
    size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_paged_attention_decode_int8 with the launch plan that
 * pkv_paged_attention_plan left in `workspace` for the same sizes (the plan
 * does not depend on the cache's element type): same arguments, semantics
 * and results; the decision of when each sequence starts (and, for -5, the
 * sibling groups) is read from the plan instead of made in the call. A
 * workspace without a plan of this batch flags PKV_DEV_BAD_PLAN and runs
 * every sequence in natural order, still computing every output.
 */
pkv_status_t pkv_paged_attention_decode_int8_planned(
    void* out, const void* q, const int8_t* k_cache, const int8_t* v_cache,
    const float* k_scale, const float* v_scale, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
    int head_dim, int max_blocks_per_seq, int num_blocks, float scale,
    pkv_dtype_t dtype, int partition_size, void* workspace,
    size_t workspace_bytes, pkv_stream_t stream);

/*
 * Copy-on-write block copies of an INT8 cache: like pkv_copy_blocks, block
 * src of the codes and of the scales (K and V) is copied to block dst.
 */
pkv_status_t pkv_copy_blocks_int8(
    int8_t* k_cache, int8_t* v_cache, float* k_scale, float* v_scale,
    const int64_t* src_dst_pairs, int num_pairs, int num_kv_heads, int head_dim,
    int num_blocks, pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Host block manager ([S] "KV キャッシュマネージャ", [B] "OSの知恵をGPUへ")  */
/* ------------------------------------------------------------------------ */
/*
 * Host memory only; not thread-safe (one handle per thread or external lock).
 * Free list: a stack, initially initial_free_order (index 0 at the bottom)
 * or 0..num_blocks-1; allocation pops the top; a block whose refcount drops
 * to 0 is pushed back. Within a call, blocks are taken in logical order and
 * returned in table order. Every failing call leaves the state unchanged.
 */
typedef struct pkv_bm pkv_bm_t;

/* block_size must be 16. initial_free_order: NULL or a permutation of
 * 0..num_blocks-1 (host). */
pkv_status_t pkv_bm_create(int num_blocks, int block_size,
                           const int32_t* initial_free_order, pkv_bm_t** out);
void pkv_bm_destroy(pkv_bm_t* bm);

/* New sequence holding num_tokens tokens: ceil(num_tokens/16) fresh blocks. */
pkv_status_t pkv_bm_add_seq(pkv_bm_t* bm, int64_t seq_id, int64_t num_tokens);

/* child shares every block of parent (refcount + 1 each); no data moves
 * ([B]: sharing by reference count only). */
pkv_status_t pkv_bm_fork(pkv_bm_t* bm, int64_t parent, int64_t child);

/*
 * Reserves the slot of the sequence's next token. With L tokens:
 *  - L % 16 == 0: a new block is appended;
 *  - else if the last block is shared (refcount > 1): copy-on-write -- a new
 *    block replaces it in this table, the old block's refcount drops by one,
 *    and (*cow_src_out, *cow_dst_out) = (old, new) must be copied with
 *    pkv_copy_blocks before the new token is written;
 *  - else the token goes into the last block in place.
 * *slot_out = table[L/16]*16 + L%16; the length becomes L+1. The CoW outputs
 * are -1 when no copy is needed.
 */
pkv_status_t pkv_bm_append_slot(pkv_bm_t* bm, int64_t seq_id, int64_t* slot_out,
                                int64_t* cow_src_out, int64_t* cow_dst_out);

/* append_slot for n sequences in order, all-or-nothing. slots_out[n];
 * pairs_out[n][2] receives the copy pairs packed at the front and
 * *num_pairs_out their count. */
pkv_status_t pkv_bm_append_slots(pkv_bm_t* bm, const int64_t* seq_ids, int n,
                                 int64_t* slots_out, int64_t* pairs_out,
                                 int* num_pairs_out);

/* Drop the sequence; blocks whose refcount reaches 0 return to the free list. */
pkv_status_t pkv_bm_free_seq(pkv_bm_t* bm, int64_t seq_id);

/*
 * Beam search step ([S] "並列サンプリングやビームサーチでの共有": beams share
 * blocks and copy a shared block only when a write reaches it): new beam i
 * (id new_ids[i]) continues old beam old_ids[parents[i]] -- it takes a copy of
 * that beam's table and length, each live block's refcount + 1 -- and then
 * every old beam is dropped (in the given order, blocks in table order;
 * blocks whose refcount reaches 0 return to the free list). Beams of beams
 * nest to any depth. old_ids must be distinct live sequences; new_ids
 * distinct, each either unused or one of old_ids. Allocates nothing, so it
 * never runs out of blocks; the next pkv_bm_append_slots emits the copies.
 * Host memory; all-or-nothing (PKV_ERR_INVALID_ARG leaves the state as is).
 */
pkv_status_t pkv_bm_beam_reorder(pkv_bm_t* bm, const int64_t* old_ids, int num_old,
                                 const int32_t* parents, const int64_t* new_ids,
                                 int num_new);

/*
 * Block-granular prefix sharing across requests (the shared-prefix workloads
 * of [S]; sharing by reference count, [B] "OSの知恵をGPUへ"): a new sequence
 * of num_tokens tokens whose first prefix_tokens tokens repeat those of
 * sequence `donor`. The whole blocks of that common prefix,
 * n = min(prefix_tokens, num_tokens, donor length) / 16 (rounded down), are
 * shared with the donor (refcount + 1); ceil(num_tokens/16) - n fresh blocks
 * follow. *shared_tokens_out (may be NULL) = 16 * n: the caller writes K/V
 * for positions from there on. PKV_ERR_OUT_OF_BLOCKS if the fresh blocks are
 * not free; PKV_ERR_INVALID_ARG for an existing seq_id, an unknown donor or a
 * prefix block the donor has released. All-or-nothing.
 */
pkv_status_t pkv_bm_add_seq_with_prefix(pkv_bm_t* bm, int64_t seq_id, int64_t num_tokens,
                                        int64_t donor, int64_t prefix_tokens,
                                        int64_t* shared_tokens_out);

/*
 * Sliding window ([G] "他のKVキャッシュ最適化との組み合わせ": sliding-window
 * attention combined with paging): drops the sequence's hold on every block
 * wholly before position first_token (table entries j with
 * (j+1)*16 <= first_token), in table order. Those entries become -1, so later
 * blocks keep their logical indices; a block whose refcount reaches 0 returns
 * to the free list. With window W, first_token = max(0, L - W) releases
 * exactly the blocks pkv_paged_attention_decode_sliding never reads.
 * first_token must lie in [0, length]. *released_out (may be NULL) receives
 * the number of entries dropped; released entries are skipped by fork and
 * free_seq.
 */
pkv_status_t pkv_bm_release_before(pkv_bm_t* bm, int64_t seq_id, int64_t first_token,
                                   int* released_out);

/* Padded block tables and lengths of n sequences (host buffers):
 * table_out[n][max_blocks_per_seq] (-1 padded), lens_out[n]. */
pkv_status_t pkv_bm_block_tables(const pkv_bm_t* bm, const int64_t* seq_ids, int n,
                                 int max_blocks_per_seq, int32_t* table_out,
                                 int32_t* lens_out);

pkv_status_t pkv_bm_refcount(const pkv_bm_t* bm, int block, int32_t* out);
pkv_status_t pkv_bm_seq_len(const pkv_bm_t* bm, int64_t seq_id, int64_t* out);
int pkv_bm_num_free(const pkv_bm_t* bm);
int pkv_bm_num_seqs(const pkv_bm_t* bm);
/* Copies the free stack (bottom first) into out[capacity]; returns its size. */
int pkv_bm_free_stack(const pkv_bm_t* bm, int32_t* out, int capacity);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H_ */
