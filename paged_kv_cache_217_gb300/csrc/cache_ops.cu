// reshape_and_cache and copy_blocks: bit copies with 16-byte vectors; the
// INT8 cache write, which quantises each row on its way into the pool.
//
// reshape_and_cache writes each decode step's new K/V row into its slot, the
// "fill the last block" step of the KV cache manager (abeam.tech summary of
// "Efficient Memory Management for Large Language Model Serving with
// PagedAttention", section "KV キャッシュマネージャ"). copy_blocks is the
// copy-on-write duplication of a shared block (same summary, section
// "並列サンプリングやビームサーチでの共有"; glossary entry
// "PagedAttention（ページドアテンション）", "コピーオンライト（Copy-on-Write）共有").
// Both are HBM-bound copies; each thread moves 16-byte vectors, consecutive
// threads consecutive vectors, so loads and stores are fully coalesced.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "decode.cuh"
#include "device_common.cuh"
#include "launch.h"

namespace pkv {
namespace {

// One thread per 16-byte vector of a (token, KV head) row.
__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                         uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                         const int64_t* __restrict__ slots, int64_t total, int num_kv_heads,
                         int vec_per_row, int64_t num_slots, unsigned int* status) {
  // The decode kernel that usually follows may become resident now; it waits
  // for this grid to finish before reading the pools.
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int c = int(i % vec_per_row);
  const int64_t tg = i / vec_per_row;
  const int gh = int(tg % num_kv_heads);
  const int64_t t = tg / num_kv_heads;
  // the row and its slot are independent loads: both in flight at once
  const int64_t slot = __ldg(slots + t);
  const uint4 kx = __ldg(k + i), vx = __ldg(v + i);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (gh == 0 && c == 0) flag(status, PKV_DEV_BAD_SLOT);
    return;
  }
  const int64_t blk = slot / kBlock, off = slot % kBlock;
  const int64_t dst = ((blk * num_kv_heads + gh) * kBlock + off) * vec_per_row + c;
  k_pool[dst] = kx;
  v_pool[dst] = vx;
}

// ---- INT8 cache write ---------------------------------------------------
// One warp per (token, KV head) row of K and of V: each lane holds D/32
// consecutive elements; the warp's max |x| gives the row scale
// s = max|x| / 127 and the codes rint(x / s) (IEEE division, ties to even),
// both decisions taken in fp32 exactly as the definition states.
template <typename T>
__device__ __forceinline__ float elem_to_float(T x);
template <>
__device__ __forceinline__ float elem_to_float<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float elem_to_float<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <int BYTES>
struct Chunk;  // a register chunk of BYTES bytes
template <> struct Chunk<2> { using type = unsigned short; };
template <> struct Chunk<4> { using type = uint32_t; };
template <> struct Chunk<8> { using type = uint2; };
template <> struct Chunk<16> { using type = uint4; };

template <typename T, int D>
using RowChunk = typename Chunk<D / 32 * 2>::type;  // one lane's D/32 elements of a row

template <typename T, int D>
__device__ __forceinline__ RowChunk<T, D> load_row_chunk(const T* __restrict__ src, int lane) {
  return __ldg(reinterpret_cast<const RowChunk<T, D>*>(src) + lane);
}

template <typename T, int D>
__device__ __forceinline__ void quantize_row(const RowChunk<T, D>& raw, int8_t* __restrict__ codes,
                                             float* __restrict__ scale, int lane) {
  constexpr int E = D / 32;  // elements per lane
  using Out = typename Chunk<E>::type;
  const T* xs = reinterpret_cast<const T*>(&raw);
  float x[E];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    x[i] = elem_to_float(xs[i]);
    m = fmaxf(m, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  const float s = __fdiv_rn(m, 127.f);
  Out packed;
  unsigned char* pb = reinterpret_cast<unsigned char*>(&packed);
#pragma unroll
  for (int i = 0; i < E; ++i) {
    int c = 0;
    if (s > 0.f) c = min(127, max(-127, __float2int_rn(__fdiv_rn(x[i], s))));
    pb[i] = static_cast<unsigned char>(c & 0xff);
  }
  reinterpret_cast<Out*>(codes)[lane] = packed;
  if (lane == 0) *scale = s;
}

template <typename T, int D>
__global__ void __launch_bounds__(256)
reshape_and_cache_int8_kernel(const T* __restrict__ k, const T* __restrict__ v, int8_t* __restrict__ k_codes,
                              int8_t* __restrict__ v_codes, float* __restrict__ k_scale,
                              float* __restrict__ v_scale, const int64_t* __restrict__ slots, int64_t rows,
                              int num_kv_heads, int64_t num_slots, unsigned int* status) {
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // warp-uniform
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int gh = int(row % num_kv_heads);
  const int64_t t = row / num_kv_heads;
  // the rows and their slot are independent loads: all in flight at once
  const int64_t slot = __ldg(slots + t);
  const RowChunk<T, D> kx = load_row_chunk<T, D>(k + row * D, lane);
  const RowChunk<T, D> vx = load_row_chunk<T, D>(v + row * D, lane);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (gh == 0 && lane == 0) flag(status, PKV_DEV_BAD_SLOT);
    return;
  }
  const int64_t dst = ((slot / kBlock) * num_kv_heads + gh) * kBlock + slot % kBlock;  // pool row
  quantize_row<T, D>(kx, k_codes + dst * D, k_scale + dst, lane);
  quantize_row<T, D>(vx, v_codes + dst * D, v_scale + dst, lane);
}

template <typename T, int D>
cudaError_t launch_int8_write(const void* k, const void* v, int8_t* kc, int8_t* vc, float* ks, float* vs,
                              const int64_t* slots, int64_t rows, int num_kv_heads, int64_t num_slots,
                              unsigned int* status, cudaStream_t stream) {
  const int64_t nblk = (rows + 7) / 8;  // 8 warps (rows) per CTA
  reshape_and_cache_int8_kernel<T, D><<<unsigned(nblk), 256, 0, stream>>>(
      static_cast<const T*>(k), static_cast<const T*>(v), kc, vc, ks, vs, slots, rows, num_kv_heads, num_slots,
      status);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_int8_write_t(const void* k, const void* v, int8_t* kc, int8_t* vc, float* ks, float* vs,
                                const int64_t* slots, int64_t rows, int num_kv_heads, int head_dim,
                                int64_t num_slots, unsigned int* status, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_int8_write<T, 64>(k, v, kc, vc, ks, vs, slots, rows, num_kv_heads, num_slots, status, stream);
    case 128: return launch_int8_write<T, 128>(k, v, kc, vc, ks, vs, slots, rows, num_kv_heads, num_slots, status, stream);
    case 256: return launch_int8_write<T, 256>(k, v, kc, vc, ks, vs, slots, rows, num_kv_heads, num_slots, status, stream);
    default: return cudaErrorInvalidValue;
  }
}

constexpr int kCopyThreads = 256;
constexpr int kCopyVecPerThread = 4;

// grid.y = pair; grid.x strides over the block's 16-byte vectors (all KV heads).
__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                   const int64_t* __restrict__ pairs, int64_t vec_per_block, int num_blocks,
                   unsigned int* status) {
  const int p = blockIdx.y;
  const int64_t src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(status, PKV_DEV_BAD_PAIR);
    return;
  }
  const uint4* ks = k_pool + src * vec_per_block;
  const uint4* vs = v_pool + src * vec_per_block;
  uint4* kd = k_pool + dst * vec_per_block;
  uint4* vd = v_pool + dst * vec_per_block;
  const int64_t base = int64_t(blockIdx.x) * kCopyThreads * kCopyVecPerThread + threadIdx.x;
  uint4 kr[kCopyVecPerThread], vr[kCopyVecPerThread];
#pragma unroll
  for (int u = 0; u < kCopyVecPerThread; ++u) {
    const int64_t i = base + int64_t(u) * kCopyThreads;
    if (i < vec_per_block) {
      kr[u] = ks[i];
      vr[u] = vs[i];
    }
  }
#pragma unroll
  for (int u = 0; u < kCopyVecPerThread; ++u) {
    const int64_t i = base + int64_t(u) * kCopyThreads;
    if (i < vec_per_block) {
      kd[i] = kr[u];
      vd[i] = vr[u];
    }
  }
}

// Self-test of the bounded wait: arms an mbarrier for 16 bytes that no copy
// will deliver and waits on it exactly as the decode kernels wait on a tile,
// with a short limit. The wait runs out and the status word gets
// PKV_DEV_WAIT_TIMEOUT; nothing is in flight, so the CTA exits cleanly.
__global__ void bounded_wait_selftest_kernel(unsigned long long limit_ns, unsigned int* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_init_fence();
    mbar_arrive_expect_tx(b, 16);
  }
  __syncwarp();
  const bool ok = mbar_wait_bounded(b, 0, limit_ns);
  if (!__all_sync(kFull, ok) && threadIdx.x == 0) flag(status, PKV_DEV_WAIT_TIMEOUT);
}

// The launch plan of a batch: its long-first order (grid row -> sequence),
// computed once for every decode grid that takes it. The buckets of
// order_bucket -- long sequences, the rest and, with short_last, short
// sequences -- each in natural order, into order[S], then the plan's header
// {kPlanMagic, S, 0, 0}, which the decode kernels check before they use the
// order. One CTA, one thread per sequence (S <= 1024). Launched with
// programmatic dependent launch: it lets a decode grid that follows become
// resident at once, reads only the lengths (which no kernel of this library
// writes), and waits for its own predecessor before it exits, so its
// completion implies that predecessor's.
__global__ void __launch_bounds__(1024)
seq_order_kernel(const int32_t* __restrict__ lens, int S, int max_len, int window, int short_last,
                 int32_t* __restrict__ order, int4* __restrict__ header, const int32_t* __restrict__ tables,
                 int max_blocks, int4* __restrict__ rows) {
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ long long part_tiles[32];
  __shared__ int part_long[32], part_rest[32], part_short[32];
  const int s = threadIdx.x, lane = s & 31, warp = s >> 5;
  int tiles = 0, raw_len = 0;
  if (s < S) {
    int L = __ldg(lens + s);
    raw_len = L;
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    if (window > 0 && L > window) L = window;
    tiles = (L + kBlock - 1) / kBlock;
  }
  long long t = tiles;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
  if (lane == 0) part_tiles[warp] = t;
  __syncthreads();
  long long total = 0;
  for (int w = 0; w < int(blockDim.x >> 5); ++w) total += part_tiles[w];
  const int b = s < S ? order_bucket(tiles, S, total, short_last != 0) : -1;
  const unsigned lb = __ballot_sync(kFull, b == 0), rb = __ballot_sync(kFull, b == 1),
                 sb = __ballot_sync(kFull, b == 2);
  if (lane == 0) {
    part_long[warp] = __popc(lb);
    part_rest[warp] = __popc(rb);
    part_short[warp] = __popc(sb);
  }
  __syncthreads();
  const unsigned below = (1u << lane) - 1u;
  int long_before = __popc(lb & below), rest_before = __popc(rb & below), short_before = __popc(sb & below);
  int n_long = 0, n_rest = 0;
  for (int w = 0; w < int(blockDim.x >> 5); ++w) {
    if (w < warp) {
      long_before += part_long[w];
      rest_before += part_rest[w];
      short_before += part_short[w];
    }
    n_long += part_long[w];
    n_rest += part_rest[w];
  }
  if (s < S) {
    const int rank = b == 0 ? long_before : (b == 1 ? n_long + rest_before : n_long + n_rest + short_before);
    order[rank] = s;
    if (rows) {  // the row of this rank: the sequence, its length and first six block ids (none without tables)
      int id[6];
#pragma unroll
      for (int i = 0; i < 6; ++i) id[i] = tables && i < max_blocks ? __ldg(tables + size_t(s) * max_blocks + i) : -1;
      rows[2 * rank] = make_int4(tables ? s : -1, raw_len, id[0], id[1]);
      rows[2 * rank + 1] = make_int4(id[2], id[3], id[4], id[5]);
    }
  }
  if (s == 0) *header = make_int4(kPlanMagic, S, 0, 0);
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Inclusive scan (sum, or max with MAX) over the threads of a CTA of up to
// 1024 threads; every thread calls it. Warp 0 scans the warps' totals.
template <bool MAX>
__device__ __forceinline__ int cta_inclusive_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = int(blockDim.x >> 5);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v = MAX ? max(v, n) : v + n;
  }
  __syncthreads();  // earlier readers of warp_tot are done
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int x0 = lane < nwarps ? warp_tot[lane] : (MAX ? INT_MIN : 0);
    int x = x0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x = MAX ? max(x, n) : x + n;
    }
    const int before = __shfl_up_sync(kFull, x, 1);  // the scan of the warps before this lane's
    if (lane < nwarps) warp_tot[lane] = lane == 0 ? (MAX ? INT_MIN : 0) : before;
  }
  __syncthreads();
  return MAX ? max(v, warp_tot[warp]) : v + warp_tot[warp];
}

// The prefix plan of a batch for the shared-prefix schedule
// (decode_prefix.cuh).
//  * Groups: for each sequence s > 0, lcp[s] = the number of whole blocks at
//    the start of its table that hold the same physical ids as its
//    predecessor's (at most the whole blocks of either length). Sequence s
//    continues its predecessor's run when lcp[s] >= min_blocks; runs are cut
//    into groups of at most max_members, each sharing the smallest lcp P of
//    its links. A group's work is its tiles: P shared ones, then each
//    member's own.
//  * Chunks: when the grid (groups and other sequences, times Hkv) is less
//    than one wave of `slots` (CTAs the decode grid holds at once), a group
//    is split into parts = ceil(work / c) chunks (1..kPrefixMaxParts), c =
//    max(kPrefixMinChunk, W x Hkv / slots) for W the batch's tiles (groups
//    counted as above, other sequences whole); else every group is one
//    chunk. A part is a range of block indices [jb, je) of equal work;
//    chunks are written longest first (LPT), a group's parts together.
//  * Others: the sequences outside any group, in batch order.
// Writes groups {first, members, P, parts} (batch order), chunks {group,
// part, jb, je}, others, the header {kPlanMagicPrefix, S, chunks, others},
// and zeroes the merge counters [S][Hkv]. One CTA of 1024 threads, S <= 1024,
// tables of at most kPrefixMaxBlocks blocks; launched like seq_order_kernel.
__global__ void __launch_bounds__(1024)
prefix_plan_kernel(const int32_t* __restrict__ lens, const int32_t* __restrict__ tables, int S, int max_blocks,
                   int Hkv, int slots, int min_blocks, int max_members, int4* __restrict__ header,
                   int4* __restrict__ groups, int4* __restrict__ chunks, int32_t* __restrict__ others,
                   unsigned int* __restrict__ counters) {
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ int slen[kOrderMaxSeqs];       // clamped lengths
  __shared__ int lcp[kOrderMaxSeqs];
  __shared__ int cwork[kOrderMaxSeqs / 2];  // per group: tiles of one chunk
  __shared__ int rparts[kOrderMaxSeqs / 2]; // per rank: parts of the group of that rank
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x;
  const int max_len = max_blocks * kBlock;
  for (int s = tid; s < S; s += blockDim.x) {
    int L = __ldg(lens + s);
    slen[s] = L < 0 ? 0 : (L > max_len ? max_len : L);
  }
  for (int i = tid; i < S * Hkv; i += blockDim.x) counters[i] = 0u;
  __syncthreads();
  for (int s = tid; s < S; s += blockDim.x) lcp[s] = s > 0 ? min(slen[s], slen[s - 1]) / kBlock : 0;
  __syncthreads();
  // lcp: every table entry j < lcp[s] of every sequence at once (one pass of
  // loads), the first mismatch with the predecessor's entry kept by atomicMin
  const int entries = S * max_blocks;
  constexpr int U = 8;  // entries a thread has in flight
  for (int i0 = tid; i0 < entries; i0 += U * int(blockDim.x)) {
    int x[U], y[U], si[U], ji[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * int(blockDim.x);
      si[u] = i < entries ? i / max_blocks : 0;
      ji[u] = i - si[u] * max_blocks;
      const bool on = i < entries && si[u] > 0 && ji[u] < lcp[si[u]];
      const int32_t* ra = tables + size_t(si[u]) * max_blocks + ji[u];
      x[u] = on ? __ldg(ra) : 0;
      y[u] = on ? __ldg(ra - max_blocks) : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (x[u] != y[u]) atomicMin(&lcp[si[u]], ji[u]);
  }
  __syncthreads();
  // the start of each sequence's run: an inclusive max-scan of (s if it starts a run, else -1)
  const int s = tid;
  const bool in_batch = s < S;
  const bool link = in_batch && s > 0 && lcp[s] >= min_blocks;
  const int run_start = cta_inclusive_scan<true>((in_batch && !link) ? s : -1, warp_tot);
  // group leaders: every max_members-th sequence of a run; a sequence is in a
  // group unless it leads one of a single member
  const int lead = in_batch ? run_start + (s - run_start) / max_members * max_members : 0;
  const bool grouped = in_batch && (s != lead || (s + 1 < S && lcp[s + 1] >= min_blocks));
  int members = 0, shared = 0, work = 0, tiles[kPrefixRows];
  if (in_batch && s == lead && grouped) {
    members = 1;
    shared = kPrefixMaxBlocks;
    while (members < max_members && s + members < S && lcp[s + members] >= min_blocks) {
      shared = min(shared, lcp[s + members]);
      ++members;
    }
  }
  const bool leader = members >= 2;
  if (leader) {
    work = shared;
#pragma unroll
    for (int m = 0; m < kPrefixRows; ++m) {
      tiles[m] = m < members ? (slen[s + m] + kBlock - 1) / kBlock : 0;
      if (m < members) work += tiles[m] - shared;
    }
  } else if (in_batch && !grouped) {
    work = (slen[s] + kBlock - 1) / kBlock;
  }
  // group index (leaders before this one), other-sequence index, batch tiles
  const int gi = cta_inclusive_scan<false>(leader ? 1 : 0, warp_tot) - (leader ? 1 : 0);
  __shared__ int totals[3];
  if (tid == blockDim.x - 1) totals[0] = gi + (leader ? 1 : 0);
  const int oi = cta_inclusive_scan<false>((in_batch && !grouped) ? 1 : 0, warp_tot) - ((in_batch && !grouped) ? 1 : 0);
  if (tid == blockDim.x - 1) totals[1] = oi + ((in_batch && !grouped) ? 1 : 0);
  const int wsum = cta_inclusive_scan<false>(work, warp_tot);
  if (tid == blockDim.x - 1) totals[2] = wsum;
  __syncthreads();
  const int G = totals[0], n_others = totals[1];
  const int64_t W = totals[2];
  if (in_batch && !grouped) others[oi] = s;
  // parts: only a grid of less than one wave of resident CTAs splits groups,
  // into chunks of about one wave's share of the batch's tiles
  const int sl = slots > 0 ? slots : 1;
  const bool split = int64_t(G + n_others) * Hkv < sl;
  const int c = int(max(int64_t(kPrefixMinChunk), (W * Hkv + sl - 1) / sl));
  int parts = leader ? (split ? min(kPrefixMaxParts, (work + c - 1) / c) : 1) : 0;
  // at most S chunks: groups are at most S / 2, so two parts a group always fit
  const int psum = cta_inclusive_scan<false>(parts, warp_tot);
  if (tid == blockDim.x - 1) totals[2] = psum;
  __syncthreads();
  if (totals[2] > S) parts = min(parts, 2);
  if (leader) cwork[gi] = (work + parts - 1) / parts;
  __syncthreads();
  // rank of this group by chunk work (longest first, ties in batch order)
  int rank = 0;
  if (leader) {
    const int w = cwork[gi];
    for (int j = 0; j < G; ++j) {
      const int x = cwork[j];
      rank += (x > w || (x == w && j < gi)) ? 1 : 0;
    }
    rparts[rank] = parts;
  }
  __syncthreads();
  const int rp = tid < G ? rparts[tid] : 0;
  const int rincl = cta_inclusive_scan<false>(rp, warp_tot);
  __syncthreads();
  if (tid < G) cwork[tid] = rincl - rp;  // chunk index of the first part of the group of rank tid
  if (tid == blockDim.x - 1) totals[0] = rincl;
  __syncthreads();
  const int nchunks = totals[0];
  if (leader) {
    groups[gi] = make_int4(s, members, shared, parts);
    const int base = cwork[rank];
    int maxn = shared;
#pragma unroll
    for (int m = 0; m < kPrefixRows; ++m)
      if (m < members) maxn = max(maxn, tiles[m]);
    // F(j): work of blocks [0, j); part q starts at the first j with F(j) >= floor(q * work / parts)
    auto F = [&](int j) {
      int f = min(j, shared);
#pragma unroll
      for (int m = 0; m < kPrefixRows; ++m)
        if (m < members) f += max(0, min(tiles[m], j) - shared);
      return f;
    };
    int jb = 0;
    for (int q = 0; q < parts; ++q) {
      int je = maxn;
      if (q + 1 < parts) {
        const int target = int(int64_t(q + 1) * work / parts);
        int lo = jb, hi = maxn;  // the first j in [lo, hi] with F(j) >= target
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (F(mid) >= target) hi = mid; else lo = mid + 1;
        }
        je = lo;
      }
      chunks[base + q] = make_int4(gi, q, jb, je);
      jb = je;
    }
  }
  if (tid == 0) *header = make_int4(kPlanMagicPrefix, S, nchunks, n_others);
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t launch_seq_order(const int32_t* lens, int num_seqs, int max_len, int window, bool short_last,
                             int4* plan, const int32_t* tables, int max_blocks, int4* rows, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(unsigned((num_seqs + 31) / 32 * 32));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int32_t* order = reinterpret_cast<int32_t*>(plan + 1);
  return cudaLaunchKernelEx(&cfg, seq_order_kernel, lens, num_seqs, max_len, window, short_last ? 1 : 0, order, plan,
                            tables, max_blocks, rows);
}

cudaError_t launch_prefix_plan(const int32_t* lens, const int32_t* tables, int num_seqs, int max_blocks,
                               int num_kv_heads, int slots, int max_members, int4* header, int4* groups, int4* chunks,
                               int32_t* others, unsigned int* counters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefix_plan_kernel, lens, tables, num_seqs, max_blocks, num_kv_heads, slots,
                            kPrefixMinBlocks, max_members, header, groups, chunks, others, counters);
}

namespace {
__global__ void trace_stamp_kernel(unsigned long long* dst) { *dst = global_timer_ns(); }
}  // namespace

cudaError_t launch_trace_stamp(unsigned long long* dst, cudaStream_t stream) {
  trace_stamp_kernel<<<1, 1, 0, stream>>>(dst);
  return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(unsigned long long limit_ns, unsigned int* status, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                                     const int64_t* slots, int num_tokens, int num_kv_heads,
                                     int head_dim, int num_blocks, unsigned int* status,
                                     cudaStream_t stream) {
  const int vec_per_row = head_dim / 8;
  const int64_t total = int64_t(num_tokens) * num_kv_heads * vec_per_row;
  if (total == 0) return cudaSuccess;
  const int64_t nblk = (total + 255) / 256;
  reshape_and_cache_kernel<<<unsigned(nblk), 256, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(k_pool),
      static_cast<uint4*>(v_pool), slots, total, num_kv_heads, vec_per_row,
      int64_t(num_blocks) * kBlock, status);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache_int8(const void* k, const void* v, bool bf16, int8_t* k_codes,
                                          int8_t* v_codes, float* k_scale, float* v_scale, const int64_t* slots,
                                          int num_tokens, int num_kv_heads, int head_dim, int num_blocks,
                                          unsigned int* status, cudaStream_t stream) {
  const int64_t rows = int64_t(num_tokens) * num_kv_heads;
  if (rows == 0) return cudaSuccess;
  const int64_t num_slots = int64_t(num_blocks) * kBlock;
  return bf16 ? launch_int8_write_t<__nv_bfloat16>(k, v, k_codes, v_codes, k_scale, v_scale, slots, rows,
                                                   num_kv_heads, head_dim, num_slots, status, stream)
              : launch_int8_write_t<__half>(k, v, k_codes, v_codes, k_scale, v_scale, slots, rows, num_kv_heads,
                                            head_dim, num_slots, status, stream);
}

cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int64_t* pairs, int num_pairs,
                               int num_kv_heads, int head_dim, int num_blocks,
                               unsigned int* status, cudaStream_t stream) {
  return launch_copy_blocks_bytes(k_pool, v_pool, pairs, num_pairs, int64_t(num_kv_heads) * kBlock * head_dim * 2,
                                  num_blocks, status, stream);
}

cudaError_t launch_copy_blocks_bytes(void* k_pool, void* v_pool, const int64_t* pairs, int num_pairs,
                                     int64_t bytes_per_block, int num_blocks, unsigned int* status,
                                     cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t vec_per_block = bytes_per_block / 16;
  const int64_t per_cta = int64_t(kCopyThreads) * kCopyVecPerThread;
  const dim3 grid(unsigned((vec_per_block + per_cta - 1) / per_cta), unsigned(num_pairs));
  copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(static_cast<uint4*>(k_pool),
                                                        static_cast<uint4*>(v_pool), pairs,
                                                        vec_per_block, num_blocks, status);
  return cudaGetLastError();
}

}  // namespace pkv
