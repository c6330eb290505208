// PagedAttention decode kernels (sm_103a).
//
// What is computed: for each sequence s and query head h, ordinary softmax
// attention of q[s][h] over the sequence's L tokens, whose K/V rows are
// reached through the block table: position p lives in physical block
// block_tables[s][p/16], slot p%16. This is the PagedAttention kernel of the
// abeam.tech summary of "Efficient Memory Management for Large Language Model
// Serving with PagedAttention" (section "技術の仕組み": the kernel walks the
// block table to read non-contiguous KV; "よくある質問": the attention formula
// itself is unchanged), with the block layout of the glossary entry
// "PagedAttention（ページドアテンション）" ("PagedAttentionの解決策").
//
// How (none of this is on the pages; it is this library's GB300 design):
//  * One CTA per (sequence, KV head, partition): the G query heads of a GQA
//    group share every K/V tile they read, so KV is read from HBM once.
//  * One (block, KV head) tile of K (or V) is a contiguous 16*D*2-byte span,
//    so a single untiled bulk copy (TMA engine, cp.async.bulk) moves it into
//    shared memory; only the tile's valid rows are copied.
//  * Each warp owns a private ring of STAGES (K, V) stages with one mbarrier
//    each and processes tiles warp, warp+NW, ...; its lane 0 keeps the ring
//    full. Warps never wait for each other until the final merge.
//  * Lanes split each 16-row tile as RPP rows x LPR lanes per row, 16 bytes
//    (8 elements) per lane. Dot products are reduced across the LPR lanes of
//    a row with a butterfly reduce-scatter, so each lane ends up owning a few
//    (row, head) scores instead of every lane reducing every score.
//  * Online softmax in fp32 in the log2 domain (q is pre-scaled by
//    scale*log2 e, exponentials use ex2.approx): running max m, running sum
//    l, running weighted V sum; the accumulator is rescaled only when a
//    head's max grows.
//  * Warps are merged through shared memory (the same max/sum rescaling).
//  * Split-K: each partition writes (m, l, unnormalised o) in fp32; the last
//    CTA of a (sequence, KV head) to finish -- counted by an atomic counter in
//    the workspace, which it resets -- merges them by log-sum-exp. Sequences
//    that fit in one partition are finished by their CTA directly.
//  * The KV storage format is a policy of the tile math: 16-bit elements
//    (KvHalf) or int8 codes with one fp32 scale per row (KvInt8).
//  * A sliding window of W tokens starts the tiles at the block holding
//    position L - W and masks the rows before it (token_range).
#pragma once

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "device_common.cuh"

namespace pkv {

struct DecodeArgs {
  void* out;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale; // INT8 cache: per-row scales [num_blocks][Hkv][16] (else unused)
  const float* v_scale;
  float* part_o;        // split-K: [S][Hq][max_parts][D] unnormalised sums
  float2* part_ml;      // split-K: [S][Hq][max_parts] (max, sum), log2 domain
  unsigned int* counters; // split-K: [S][Hkv] partitions finished; zero between calls
  unsigned int* status; // device status word (PKV_DEV_* flags)
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;            // real query heads per KV head (<= G of the kernel)
  int max_blocks_per_seq;
  int num_blocks;
  int part_tokens;      // tokens per partition (multiple of 16)
  int max_parts;        // grid.z
  int long_first;       // start sequences of twice the mean length first (long_first_seq)
  const int32_t* order; // long_first: grid row -> sequence from a launch plan (seq_order_kernel), or null
  const int4* plan;     // the plan's header {kPlanMagic, num_seqs, 0, 0}, checked before `order` is used
  const int4* plan_rows; // launch plan rows {s, L, ids 0..5} per grid row (tensor-core one-pass grid), or null
  unsigned long long* trace;  // PKV_TRACE builds: per-CTA phase timestamps (8 words a CTA), or null
  int trace_records;          // CTAs the trace buffer holds
  int window;           // sliding window: attend over the last `window` tokens (0 = all)
  const int4* prefix_header;     // shared-prefix schedule: the prefix plan's header {magic, S, chunks, others}, or null
  const int4* prefix_groups;     // ... its groups {first member, members, shared blocks, parts}
  const int4* prefix_chunks;     // ... its chunks {group, part, first block, end block}, longest first
  const int32_t* prefix_others;  // ... the sequences outside any group
  int prefix_slots;              // ... and the grid rows reserved for chunks (num_seqs)
  float scale_log2;     // scale * log2(e)
};

// Token range a sequence of length L attends over: [first, L), with
// first = L - window for a sliding window shorter than L, else 0. The tiles
// start at the block boundary `aligned` <= first; rows before `first` in the
// first tile are masked.
struct TokenRange {
  int first, aligned;
};
__device__ __forceinline__ TokenRange token_range(int L, int window) {
  TokenRange r;
  r.first = (window > 0 && L > window) ? L - window : 0;
  r.aligned = r.first & ~(kBlock - 1);
  return r;
}

// Tracing (diagnostic builds only, -DPKV_TRACE=1): each CTA of the one-pass
// and split grid kernels records %globaltimer at its phase boundaries -- start
// (after the predecessor), sequence known, length and ids known, first tile
// landed (warp 0), tile loop done (warp 0), end -- plus its SM and (sequence,
// tiles) into a caller-supplied buffer. Off by default: no code is generated.
#ifndef PKV_TRACE
#define PKV_TRACE 0
#endif
constexpr bool kTrace = PKV_TRACE != 0;

struct TraceMarks {
  unsigned long long t[5];
};

__device__ __forceinline__ void trace_mark(TraceMarks& m, int i) {
  if constexpr (kTrace) m.t[i] = global_timer_ns();
}

__device__ __forceinline__ void trace_write(const DecodeArgs& a, const TraceMarks& m, int s, int tiles) {
  if constexpr (kTrace) {
    if (threadIdx.x != 0 || !a.trace) return;
    const unsigned long long cta = blockIdx.x + (unsigned long long)gridDim.x * (blockIdx.y + (unsigned long long)gridDim.y * blockIdx.z);
    if (cta >= (unsigned long long)a.trace_records) return;
    unsigned int smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    unsigned long long* r = a.trace + 8 * cta;
    for (int i = 0; i < 5; ++i) r[i] = m.t[i];
    r[5] = global_timer_ns();
    r[6] = smid;
    r[7] = (unsigned long long)(unsigned)s | ((unsigned long long)(unsigned)tiles << 32);
  }
}

// Waits until the kernel launched before this one in the stream has finished
// and its writes are visible (programmatic dependent launch: the grid may
// become resident while its predecessor still runs). Every global read of
// the decode kernels comes after this.
__device__ __forceinline__ void wait_for_predecessor() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Grid of the one-CTA-per-(sequence, KV head) kernels: blockIdx.x is the KV
// head (fastest in launch order, so the heads of one sequence run side by
// side), blockIdx.y the sequence's rank in the launch order, blockIdx.z the
// split-K partition.

// Batches of up to this many sequences start long sequences first.
constexpr int kOrderMaxSeqs = 1024;
// Batches of up to this many are ranked in every CTA unless planned; larger
// ones get a launch plan from a one-CTA kernel ahead of the decode grid.
constexpr int kRankInCtaMaxSeqs = 127;
// First word of a launch plan's header (pkv_paged_attention_plan).
constexpr int kPlanMagic = 0x504b5631;  // "PKV1"
// First word of a prefix plan's header (the shared-prefix schedule).
constexpr int kPlanMagicPrefix = 0x504b5831;  // "PKX1"
constexpr int kPrefixMinBlocks = 4;    // shared prefixes shorter than this stay in the members' own CTAs
constexpr int kPrefixMaxBlocks = 256;  // table widths the prefix plan compares
constexpr int kPrefixRows = 8;         // query rows per group (members x query heads per KV head)
// A group's tiles may be split over up to kPrefixMaxParts CTAs (merged by
// log-sum-exp) so that a batch of few groups still fills the GPU: only when
// the grid is under one wave of resident CTAs, in chunks of at least
// kPrefixMinChunk tiles. Measured on GB300 (LLaMA-13B beam batch, 640 group
// CTAs for 608 resident): chunks aimed at 1 or 3 waves took 61.8 and
// 67.6 us against 61.1 us unsplit -- each chunk pays a CTA's start-up and a
// merge.
constexpr int kPrefixMaxParts = 4;
constexpr int kPrefixMinChunk = 8;
// A sequence is "long" when its tile count is at least kLongFirstX2 / 2 times
// the batch mean (2x). Measured on GB300 (threshold x mean -> decode call µs):
// Llama-3-8B-shaped layer 1.5 -> 43.7, 2 -> 43.4, 2.5 -> 43.6, 4 -> 46.7;
// LLaMA-13B-shaped layer 2 -> 133.2, 2.5 -> 132.8, 3 -> 148.3.
constexpr long long kLongFirstX2 = 4;
// In launch plans of batches of 128..1024 sequences, a sequence that is not
// long is "short", and goes after all others, when its tile count is at most
// kShortLastX8 / 8 times the batch mean. Measured on
// GB300, Llama-3-8B-shaped layer (256 sequences): 0 (no short bucket) ->
// 42.9 us, 3 -> 42.2, 4 -> 41.6, 5 -> 41.3, 6 -> 41.5, 8 -> 43.2; the same
// bucket in smaller batches (the LLaMA-13B layer, the beam batch) cost
// 0.5-1.8 %, so plans of smaller batches, and the per-CTA ranking, keep two
// buckets.
constexpr long long kShortLastX8 = 5;

// Bucket of a sequence with `tiles` tiles in a batch of S sequences holding
// `total` tiles: 0 long (first), 1 the rest, 2 short (last; only with
// short_last).
__device__ __forceinline__ int order_bucket(long long tiles, int S, long long total, bool short_last) {
  if (2 * tiles * S >= kLongFirstX2 * total) return 0;
  if (short_last && kShortLastX8 > 0 && 8 * tiles * S <= kShortLastX8 * total) return 2;
  return 1;
}

// Position of the k-th (0-based) set bit of m; m has more than k set bits.
__device__ __forceinline__ int kth_set_bit(unsigned int m, int k) {
  for (int i = 0; i < k; ++i) m &= m - 1u;
  return __ffs(int(m)) - 1;
}

// The sequence that the CTAs of grid row `rank` process. Rows are dispatched
// in order, and a long sequence that starts in the last wave decides when the
// kernel ends, so sequences with at least twice the batch's mean tile count
// take the first rows (in natural order) and all others follow (in natural
// order, which keeps parallel samples of one prompt -- sequences that share
// blocks -- running side by side). Every CTA derives the same mapping from
// context_lens, so each sequence is taken exactly once. (Batches that the
// ordering kernel ranks also put their shortest sequences last.)
template <int NW>
__device__ __forceinline__ int long_first_seq(const DecodeArgs& a, int rank) {
  const int S = a.num_seqs;
  if (!a.long_first || S > kOrderMaxSeqs || S <= 1) return rank;
  if (a.order) {  // ranked once for the whole grid, by a launch plan
    const int4 h = __ldg(a.plan);
    const int s = __ldg(a.order + rank);
    if (h.x == kPlanMagic && h.y == S && s >= 0 && s < S) return s;
    // not a plan of this batch size: every CTA sees the same header and takes
    // its natural row, so each sequence is still processed exactly once
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) flag(a.status, PKV_DEV_BAD_PLAN);
    return rank;
  }
  // Batches of kRankInCtaMaxSeqs + 1 or more sequences always come with a plan
  // (the library makes one ahead of the grid), so the per-CTA ranking needs
  // room for the small batches only.
  if (S > kRankInCtaMaxSeqs) return rank;
  __shared__ int tiles[kRankInCtaMaxSeqs];
  __shared__ unsigned int long_bits[kRankInCtaMaxSeqs / 32 + 1];
  __shared__ int red[NW];
  __shared__ int picked;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int max_len = a.max_blocks_per_seq * kBlock;
  int local = 0;
  for (int s = tid; s < S; s += NW * 32) {
    int L = __ldg(a.context_lens + s);
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    if (a.window > 0 && L > a.window) L = a.window;
    tiles[s] = (L + kBlock - 1) / kBlock;
    local += tiles[s];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(kFull, local, o);
  if (lane == 0) red[warp] = local;
  __syncthreads();
  long long total = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) total += red[w];
  const int words = (S + 31) / 32;
  for (int i = warp; i < words; i += NW) {
    const int s = 32 * i + lane;
    const bool lg = s < S && order_bucket(tiles[s], S, total, false) == 0;
    const unsigned int m = __ballot_sync(kFull, lg);
    if (lane == 0) long_bits[i] = m;
  }
  __syncthreads();
  if (warp == 0) {
    // lane i owns word i (words <= 32)
    const unsigned int valid = lane < words ? (lane == words - 1 && (S & 31) ? (1u << (S & 31)) - 1u : kFull) : 0u;
    const unsigned int lb = lane < words ? long_bits[lane] : 0u;
    const int nl = __popc(lb), ns = __popc(valid & ~lb);
    int il = nl, is = ns;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(kFull, il, o), a2 = __shfl_up_sync(kFull, is, o);
      if (lane >= o) {
        il += a1;
        is += a2;
      }
    }
    const int n_long = __shfl_sync(kFull, il, 31);
    if (rank < n_long) {  // the rank-th long sequence
      if (il - nl <= rank && rank < il) picked = 32 * lane + kth_set_bit(lb, rank - (il - nl));
    } else {              // the (rank - n_long)-th other sequence
      const int r2 = rank - n_long;
      if (is - ns <= r2 && r2 < is) picked = 32 * lane + kth_set_bit(valid & ~lb, r2 - (is - ns));
    }
  }
  __syncthreads();
  return picked;
}

// Storage formats of the KV pools for the CUDA-core tile math: eight
// elements per lane per row, loaded from shared memory as floats.
template <typename T>
struct KvHalf {  // fp16 / bf16 elements
  static constexpr int ELEM = 2;
  static constexpr bool SCALED = false;
  static __device__ __forceinline__ void load8(uint32_t addr, float (&f)[8]) {
    Vec8<T>::to_float(lds128(addr), f);
  }
};

struct KvInt8 {  // int8 codes, one fp32 scale per row (16 per tile, after the codes)
  static constexpr int ELEM = 1;
  static constexpr bool SCALED = true;
  static __device__ __forceinline__ void load8(uint32_t addr, float (&f)[8]) { int8x8_to_float(lds64(addr), f); }
};

template <typename T, int D, int G, int NW, int STAGES, typename KV = KvHalf<T>>
struct DecodeCfg {
  static constexpr int LPR = D / 8;                  // lanes per row
  static constexpr int RPP = 32 / LPR;               // rows per pass
  static constexpr int NPASS = kBlock / RPP;         // passes per tile
  static constexpr int ROW_BYTES = D * KV::ELEM;
  static constexpr int TILE_BYTES = kBlock * ROW_BYTES;
  static constexpr int SCALE_BYTES = KV::SCALED ? kBlock * 4 : 0;
  // K tile, V tile, then (INT8) the 16 K scales and the 16 V scales
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES + 2 * SCALE_BYTES;
  static constexpr int V = NPASS * G;                // scores per lane before the reduction
  static constexpr int LOGV = ilog2(V);
  static constexpr int LOGL = ilog2(LPR);
  static constexpr int LOGG = ilog2(G);
  static constexpr int NH = LOGV < LOGL ? LOGV : LOGL; // halving steps
  static constexpr int NF = V >> NH;                 // scores a lane owns afterwards
  static constexpr size_t RING_BYTES = size_t(NW) * STAGES * STAGE_BYTES;
  static constexpr size_t SMEM_BYTES = RING_BYTES + size_t(NW) * STAGES * 8;
  static_assert((LPR & (LPR - 1)) == 0 && LPR >= 8 && LPR <= 32, "head_dim must be 64, 128 or 256");
  static_assert((G & (G - 1)) == 0 && G <= 8, "group size is padded to 1, 2, 4 or 8");
  static_assert(G <= LPR, "a lane's scores must belong to one head");
  static_assert(size_t(2 * G + G * D) * 4 <= size_t(STAGES) * STAGE_BYTES, "merge area fits the ring");
};

// Butterfly reduce-scatter of N per-lane partial sums across the lanes
// selected by masks M, M/2, ..., 1: each step halves the list a lane keeps
// (upper half if the lane's mask bit is set) and adds the partner's half;
// once one value is left the remaining steps are plain butterfly sums.
template <int N, int M>
struct RowReduceScatter {
  static __device__ __forceinline__ void run(float* x, int lane) {
    if constexpr (M >= 1) {
      if constexpr (N > 1) {
        const bool up = (lane & M) != 0;
#pragma unroll
        for (int j = 0; j < N / 2; ++j) {
          const float send = up ? x[j] : x[j + N / 2];
          const float keep = up ? x[j + N / 2] : x[j];
          x[j] = keep + __shfl_xor_sync(kFull, send, M);
        }
        RowReduceScatter<N / 2, M / 2>::run(x, lane);
      } else {
        x[0] += __shfl_xor_sync(kFull, x[0], M);
        RowReduceScatter<1, M / 2>::run(x, lane);
      }
    }
  }
};

// One 16-row tile: scores, online-softmax update, weighted V accumulation.
// MASK: only rows [lo, rows) of the tile are valid (the rest of the stage is
// stale or outside a sliding window).
template <typename T, int D, int G, int NW, int STAGES, bool MASK, typename KV = KvHalf<T>>
__device__ __forceinline__ void decode_tile(uint32_t kt, uint32_t vt, int lo, int rows,
                                            const float (&qf)[G][8], float (&acc)[G][8],
                                            float (&lsum)[G], float (&mrun)[G], int lane,
                                            uint32_t ksc = 0, uint32_t vsc = 0) {
  using C = DecodeCfg<T, D, G, NW, STAGES, KV>;
  constexpr int LPR = C::LPR, RPP = C::RPP, NPASS = C::NPASS, NF = C::NF;
  const int sub = lane & (LPR - 1);
  const int r = lane / LPR;

  // Partial dot products: sc[h * NPASS + i] for row i*RPP + r, this lane's 8 dims.
  float sc[C::V];
#pragma unroll
  for (int i = 0; i < NPASS; ++i) {
    float kf[8];
    KV::load8(kt + (i * RPP + r) * C::ROW_BYTES + sub * 8 * KV::ELEM, kf);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float d0 = qf[h][0] * kf[0];
      float d1 = qf[h][1] * kf[1];
      d0 = fmaf(qf[h][2], kf[2], d0);
      d1 = fmaf(qf[h][3], kf[3], d1);
      d0 = fmaf(qf[h][4], kf[4], d0);
      d1 = fmaf(qf[h][5], kf[5], d1);
      d0 = fmaf(qf[h][6], kf[6], d0);
      d1 = fmaf(qf[h][7], kf[7], d1);
      sc[h * NPASS + i] = d0 + d1;
    }
  }
  RowReduceScatter<C::V, LPR / 2>::run(sc, lane);

  // This lane now owns NF full scores of head `hl`, passes i0 .. i0+NF-1.
  const int vb = (sub >> (C::LOGL - C::NH)) << (C::LOGV - C::NH);
  const int hl = vb / NPASS;
  const int i0 = vb % NPASS;
  float mloc = -INFINITY;
#pragma unroll
  for (int e = 0; e < NF; ++e) {
    if constexpr (KV::SCALED) sc[e] *= lds_f32(ksc + ((i0 + e) * RPP + r) * 4);  // dequantise K
    if (MASK && ((i0 + e) * RPP + r < lo || (i0 + e) * RPP + r >= rows)) sc[e] = -INFINITY;
    mloc = fmaxf(mloc, sc[e]);
  }
  // Tile max of head hl: lanes that own head hl differ in the low sub bits and in r.
#pragma unroll
  for (int m = 1; m < (LPR >> C::LOGG); m <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, m));
#pragma unroll
  for (int m = LPR; m < 32; m <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, m));
  float mr = mrun[0];
#pragma unroll
  for (int h = 1; h < G; ++h)
    if (hl == h) mr = mrun[h];
  const float mnew = fmaxf(mr, mloc);
  float p[NF];
#pragma unroll
  for (int e = 0; e < NF; ++e) p[e] = fast_exp2(sc[e] - mnew);

  // Every lane learns each head's new max; rescale only heads whose max grew.
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float mn = (G == 1) ? mnew : __shfl_sync(kFull, mnew, h << (C::LOGL - C::LOGG));
    if (mn > mrun[h]) {
      const float alpha = fast_exp2(mrun[h] - mn);
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[h][c] *= alpha;
      lsum[h] *= alpha;
      mrun[h] = mn;
    }
  }

  // Weighted V: row i*RPP + r, this lane's 8 dims, every head of the group.
#pragma unroll
  for (int i = 0; i < NPASS; ++i) {
    const int row = i * RPP + r;
    float vf[8];
    KV::load8(vt + row * C::ROW_BYTES + sub * 8 * KV::ELEM, vf);
    // rows past the tile's valid ones hold stale data: their weight is 0 and
    // their values must not reach the sums (0 * NaN)
    const bool live = !MASK || (row >= lo && row < rows);
    if (MASK && !live) {
#pragma unroll
      for (int c = 0; c < 8; ++c) vf[c] = 0.f;
    }
    float vscale = 1.f;
    if constexpr (KV::SCALED) vscale = live ? lds_f32(vsc + row * 4) : 0.f;  // dequantise V via the weight
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int v = h * NPASS + i;
      const int src = r * LPR + ((v >> (C::LOGV - C::NH)) << (C::LOGL - C::NH));
      const float p_raw = __shfl_sync(kFull, p[v & (NF - 1)], src);
      lsum[h] += p_raw;
      const float pp = KV::SCALED ? p_raw * vscale : p_raw;
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[h][c] = fmaf(pp, vf[c], acc[h][c]);
    }
  }
}

// Epilogue shared by the decode kernels. On entry every warp w has published
// its running sums for the chunk in its own shared-memory area
// (smem + w * area_bytes): acc[G][D], then m[G], then l[G] (log2 domain), and
// the CTA has synchronised. The warps are merged by rescaling each to the
// common max; a sequence that fits one partition is finished here. Otherwise
// the partition's (m, l, o) go to the workspace and the last partition of the
// (sequence, KV head) to arrive merges all of them by log-sum-exp:
//   M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p.
template <typename T, int D, int G, int NW>
__device__ __forceinline__ void finish_chunk(const DecodeArgs& a, const unsigned char* smem,
                                             size_t area_bytes, int s, int g, int part, int nparts) {
  constexpr int CHUNKS = D / 8;
  const int hq0 = g * a.group;
  const bool direct = nparts == 1;
  for (int it = threadIdx.x; it < a.group * CHUNKS; it += NW * 32) {
    const int h = it / CHUNKS, c8 = it % CHUNKS;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      M = fmaxf(M, reinterpret_cast<const float*>(smem + size_t(w) * area_bytes)[G * D + h]);
    float den = 0.f, num[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) num[c] = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* ws = reinterpret_cast<const float*>(smem + size_t(w) * area_bytes);
      const float mw = ws[G * D + h];
      if (mw == -INFINITY) continue;
      const float wt = fast_exp2(mw - M);
      den = fmaf(wt, ws[G * D + G + h], den);
      const float4* src = reinterpret_cast<const float4*>(ws + h * D + c8 * 8);
      const float4 x0 = src[0], x1 = src[1];
      num[0] = fmaf(wt, x0.x, num[0]);
      num[1] = fmaf(wt, x0.y, num[1]);
      num[2] = fmaf(wt, x0.z, num[2]);
      num[3] = fmaf(wt, x0.w, num[3]);
      num[4] = fmaf(wt, x1.x, num[4]);
      num[5] = fmaf(wt, x1.y, num[5]);
      num[6] = fmaf(wt, x1.z, num[6]);
      num[7] = fmaf(wt, x1.w, num[7]);
    }
    const size_t row = size_t(s) * a.num_q_heads + hq0 + h;
    if (direct) {
      const float inv = 1.f / den;
#pragma unroll
      for (int c = 0; c < 8; ++c) num[c] *= inv;
      reinterpret_cast<uint4*>(static_cast<T*>(a.out) + row * D)[c8] = Vec8<T>::from_float(num);
    } else {
      float4* dst = reinterpret_cast<float4*>(a.part_o + (row * a.max_parts + part) * D + c8 * 8);
      dst[0] = make_float4(num[0], num[1], num[2], num[3]);
      dst[1] = make_float4(num[4], num[5], num[6], num[7]);
      if (c8 == 0) a.part_ml[row * a.max_parts + part] = make_float2(M, den);
    }
  }
  if (direct) return;

  __shared__ unsigned int last_arrival;
  __threadfence();
  __syncthreads();
  unsigned int* counter = a.counters + size_t(s) * a.num_kv_heads + g;
  if (threadIdx.x == 0) last_arrival = atomicAdd(counter, 1u) == unsigned(nparts - 1) ? 1u : 0u;
  __syncthreads();
  if (!last_arrival) return;
  __threadfence();
  for (int it = threadIdx.x; it < a.group * CHUNKS; it += NW * 32) {
    const int h = it / CHUNKS, c8 = it % CHUNKS;
    const size_t row = size_t(s) * a.num_q_heads + hq0 + h;
    const float2* ml = a.part_ml + row * a.max_parts;
    const float* po = a.part_o + row * a.max_parts * D + c8 * 8;
    float M = -INFINITY;
    for (int p = 0; p < nparts; ++p) M = fmaxf(M, __ldcg(&ml[p].x));
    float den = 0.f, num[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) num[c] = 0.f;
    for (int p = 0; p < nparts; ++p) {
      const float2 x = __ldcg(ml + p);
      const float w = fast_exp2(x.x - M);
      den = fmaf(w, x.y, den);
      const float4* src = reinterpret_cast<const float4*>(po + size_t(p) * D);
      const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
      num[0] = fmaf(w, x0.x, num[0]);
      num[1] = fmaf(w, x0.y, num[1]);
      num[2] = fmaf(w, x0.z, num[2]);
      num[3] = fmaf(w, x0.w, num[3]);
      num[4] = fmaf(w, x1.x, num[4]);
      num[5] = fmaf(w, x1.y, num[5]);
      num[6] = fmaf(w, x1.z, num[6]);
      num[7] = fmaf(w, x1.w, num[7]);
    }
    const float inv = 1.f / den;
#pragma unroll
    for (int c = 0; c < 8; ++c) num[c] *= inv;
    reinterpret_cast<uint4*>(static_cast<T*>(a.out) + row * D)[c8] = Vec8<T>::from_float(num);
  }
  if (threadIdx.x == 0) *counter = 0u;  // leave the workspace ready for the next call
}

template <typename T, int D, int G, int NW, int STAGES, typename KV = KvHalf<T>>
__global__ void __launch_bounds__(NW * 32)
paged_decode_kernel(const DecodeArgs a) {
  using C = DecodeCfg<T, D, G, NW, STAGES, KV>;
  constexpr int LPR = C::LPR;
  extern __shared__ __align__(1024) unsigned char smem[];

  wait_for_predecessor();
  TraceMarks tm{};
  trace_mark(tm, 0);
  const int g = blockIdx.x;
  const int s = long_first_seq<NW>(a, blockIdx.y), part = blockIdx.z;
  trace_mark(tm, 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & (LPR - 1), r = lane / LPR;
  const int hq0 = g * a.group;

  // Without a sliding window the first 32 block ids of this warp's tiles do
  // not depend on the length: read them together with it (entries past the
  // sequence are never used).
  int ids_early = 0;
  if (a.window == 0) {
    const int j0 = (blockIdx.z * a.part_tokens) / kBlock + warp + lane * NW;
    if (j0 < a.max_blocks_per_seq) ids_early = __ldg(a.block_tables + size_t(s) * a.max_blocks_per_seq + j0);
  }
  int L = a.context_lens[s];
  const int max_len = a.max_blocks_per_seq * kBlock;
  if (L < 0 || L > max_len) {
    if (threadIdx.x == 0 && part == 0 && g == 0) flag(a.status, PKV_DEV_BAD_CONTEXT_LEN);
    L = L < 0 ? 0 : max_len;
  }
  const TokenRange tr = token_range(L, a.window);
  const int nparts = L == 0 ? 1 : (L - tr.aligned + a.part_tokens - 1) / a.part_tokens;
  if (part >= nparts) return;
  const int pslot = part;  // partition slot of this CTA's partial in the workspace
  trace_mark(tm, 2);

  if (L == 0) {  // empty sequence: zeros
    T* o = static_cast<T*>(a.out) + (size_t(s) * a.num_q_heads + hq0) * D;
    for (int i = threadIdx.x; i < a.group * D / 8; i += NW * 32)
      reinterpret_cast<uint4*>(o)[i] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }

  const int t0 = tr.aligned + part * a.part_tokens;
  const int ntok = min(L, t0 + a.part_tokens) - t0;
  const int nb = (ntok + kBlock - 1) / kBlock;
  const int head = part == 0 ? tr.first - tr.aligned : 0;  // rows before the window in tile 0

  unsigned char* ring = smem + size_t(warp) * STAGES * C::STAGE_BYTES;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar_s = smem_addr(smem + C::RING_BYTES) + warp * STAGES * 8;
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < STAGES; ++st) mbar_init(bar_s + 8 * st, 1);
    mbar_init_fence();
  }
  __syncwarp();

  // q of this lane's 8 dims for every head of the group, in the log2 domain.
  float qf[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (h < a.group) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(
          static_cast<const T*>(a.q) + (size_t(s) * a.num_q_heads + hq0 + h) * D + sub * 8));
      Vec8<T>::to_float(u, qf[h]);
#pragma unroll
      for (int c = 0; c < 8; ++c) qf[h][c] *= a.scale_log2;
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) qf[h][c] = 0.f;
    }
  }

  // Tiles of this warp: j = warp + k*NW, k = 0 .. n_my-1. Lane k%32 of `ids`
  // holds the physical block of tile k (batches of 32, the next batch prefetched).
  const int n_my = nb > warp ? (nb - warp + NW - 1) / NW : 0;
  const int32_t* trow = a.block_tables + size_t(s) * a.max_blocks_per_seq + t0 / kBlock;
  auto load_ids = [&](int batch) -> int {
    const int k = batch * 32 + lane;
    if (k >= n_my) return 0;
    int id = __ldg(trow + warp + k * NW);
    if (id < 0 || id >= a.num_blocks) {
      flag(a.status, PKV_DEV_BAD_BLOCK_ID);
      id = 0;
    }
    return id;
  };
  int ids = 0;
  if (lane < n_my) {
    ids = a.window == 0 ? ids_early : __ldg(trow + warp + lane * NW);
    if (ids < 0 || ids >= a.num_blocks) {
      flag(a.status, PKV_DEV_BAD_BLOCK_ID);
      ids = 0;
    }
  }
  int ids_next = n_my > 32 ? load_ids(1) : 0;
  int id_batch = 0;

  const char* kbase = static_cast<const char*>(a.k_pool) + size_t(g) * C::TILE_BYTES;
  const char* vbase = static_cast<const char*>(a.v_pool) + size_t(g) * C::TILE_BYTES;
  const size_t blk_stride = size_t(a.num_kv_heads) * C::TILE_BYTES;
  // INT8: the 16 scales of tile (block, g) are 64 contiguous bytes
  const float* kscale_base = KV::SCALED ? a.k_scale + size_t(g) * kBlock : nullptr;
  const float* vscale_base = KV::SCALED ? a.v_scale + size_t(g) * kBlock : nullptr;

  auto issue = [&](int k) {  // warp-uniform; k increases by one per call
    if ((k >> 5) != id_batch) {
      ids = ids_next;
      ++id_batch;
      ids_next = (id_batch + 1) * 32 < n_my ? load_ids(id_batch + 1) : 0;
    }
    const int id = __shfl_sync(kFull, ids, k & 31);
    if (lane == 0) {
      const int j = warp + k * NW;
      const int rows = min(kBlock, ntok - j * kBlock);
      const int lo = j == 0 ? head : 0;  // rows before the window are not copied
      const uint32_t bytes = uint32_t(rows - lo) * C::ROW_BYTES;
      const uint32_t off = uint32_t(lo) * C::ROW_BYTES;
      const int st = k % STAGES;
      const uint32_t bar = bar_s + 8 * st;
      const uint32_t dst = ring_s + st * C::STAGE_BYTES;
      mbar_arrive_expect_tx(bar, 2 * bytes + 2 * C::SCALE_BYTES);
      bulk_g2s(dst + off, kbase + size_t(id) * blk_stride + off, bytes, bar);
      bulk_g2s(dst + C::TILE_BYTES + off, vbase + size_t(id) * blk_stride + off, bytes, bar);
      if constexpr (KV::SCALED) {
        const size_t so = size_t(id) * a.num_kv_heads * kBlock;
        bulk_g2s(dst + 2 * C::TILE_BYTES, kscale_base + so, C::SCALE_BYTES, bar);
        bulk_g2s(dst + 2 * C::TILE_BYTES + C::SCALE_BYTES, vscale_base + so, C::SCALE_BYTES, bar);
      }
    }
  };

  float acc[G][8], lsum[G], mrun[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    lsum[h] = 0.f;
    mrun[h] = -INFINITY;
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[h][c] = 0.f;
  }

  const int pre = n_my < STAGES ? n_my : STAGES;
  for (int k = 0; k < pre; ++k) issue(k);

  for (int k = 0; k < n_my; ++k) {
    const int st = k % STAGES;
    const uint32_t parity = (k / STAGES) & 1;
    const bool ok = mbar_wait_bounded(bar_s + 8 * st, parity);
    if (!__all_sync(kFull, ok)) {
      // A copy never completed: record it, wait (bounded) for the copies still
      // in flight into this warp's ring, and stop consuming.
      if (lane == 0) flag(a.status, PKV_DEV_WAIT_TIMEOUT);
      const int last = min(n_my, k + STAGES);
      for (int kk = k; kk < last; ++kk) mbar_wait_bounded(bar_s + 8 * (kk % STAGES), (kk / STAGES) & 1);
      break;
    }
    if (k == 0) trace_mark(tm, 3);
    const int j = warp + k * NW;
    const int rows = min(kBlock, ntok - j * kBlock);
    const int lo = j == 0 ? head : 0;
    const uint32_t kt = ring_s + st * C::STAGE_BYTES;
    const uint32_t ks = kt + 2 * C::TILE_BYTES, vs = ks + C::SCALE_BYTES;
    if (rows == kBlock && lo == 0)
      decode_tile<T, D, G, NW, STAGES, false, KV>(kt, kt + C::TILE_BYTES, 0, rows, qf, acc, lsum, mrun, lane, ks, vs);
    else
      decode_tile<T, D, G, NW, STAGES, true, KV>(kt, kt + C::TILE_BYTES, lo, rows, qf, acc, lsum, mrun, lane, ks, vs);
    __syncwarp();
    if (k + STAGES < n_my) issue(k + STAGES);
  }

  trace_mark(tm, 4);
  // Sum the row groups of the warp (lanes that differ in r).
#pragma unroll
  for (int m = LPR; m < 32; m <<= 1) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      lsum[h] += __shfl_xor_sync(kFull, lsum[h], m);
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[h][c] += __shfl_xor_sync(kFull, acc[h][c], m);
    }
  }

  // Publish the warp's (acc, m, l) in its own ring (all its copies have landed):
  // acc[G][D] first so its float4 stores stay 16-byte aligned, then m[G], l[G].
  float* wsm = reinterpret_cast<float*>(ring);
  if (r == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float4* dst = reinterpret_cast<float4*>(wsm + h * D + sub * 8);
      dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      wsm[G * D + h] = mrun[h];
      wsm[G * D + G + h] = lsum[h];
    }
  }
  __syncthreads();

  finish_chunk<T, D, G, NW>(a, smem, size_t(STAGES) * C::STAGE_BYTES, s, g, pslot, nparts);
  trace_write(a, tm, s, nb);
}

}  // namespace pkv
