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
//  * Split-K: each partition writes (m, l, unnormalised o) in fp32; the merge
//    kernel combines them by log-sum-exp. Sequences that fit in one partition
//    are finished by their CTA directly.
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
  float* part_o;        // split-K: [S][Hq][max_parts][D] unnormalised sums
  float2* part_ml;      // split-K: [S][Hq][max_parts] (max, sum), log2 domain
  unsigned int* status; // device status word (PKV_DEV_* flags)
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;            // real query heads per KV head (<= G of the kernel)
  int max_blocks_per_seq;
  int num_blocks;
  int part_tokens;      // tokens per partition (multiple of 16)
  int max_parts;        // grid.z
  float scale_log2;     // scale * log2(e)
};

template <typename T, int D, int G, int NW, int STAGES>
struct DecodeCfg {
  static constexpr int LPR = D / 8;                  // lanes per row
  static constexpr int RPP = 32 / LPR;               // rows per pass
  static constexpr int NPASS = kBlock / RPP;         // passes per tile
  static constexpr int ROW_BYTES = D * int(sizeof(T));
  static constexpr int TILE_BYTES = kBlock * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES; // K tile then V tile
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
// MASK: the tile holds only `rows` valid rows (the rest of the stage is stale).
template <typename T, int D, int G, int NW, int STAGES, bool MASK>
__device__ __forceinline__ void decode_tile(uint32_t kt, uint32_t vt, int rows,
                                            const float (&qf)[G][8], float (&acc)[G][8],
                                            float (&lsum)[G], float (&mrun)[G], int lane) {
  using C = DecodeCfg<T, D, G, NW, STAGES>;
  constexpr int LPR = C::LPR, RPP = C::RPP, NPASS = C::NPASS, NF = C::NF;
  const int sub = lane & (LPR - 1);
  const int r = lane / LPR;

  // Partial dot products: sc[h * NPASS + i] for row i*RPP + r, this lane's 8 dims.
  float sc[C::V];
#pragma unroll
  for (int i = 0; i < NPASS; ++i) {
    const uint4 u = lds128(kt + (i * RPP + r) * C::ROW_BYTES + sub * 16);
    float kf[8];
    Vec8<T>::to_float(u, kf);
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
    if (MASK && (i0 + e) * RPP + r >= rows) sc[e] = -INFINITY;
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
    uint4 u = lds128(vt + row * C::ROW_BYTES + sub * 16);
    if (MASK && row >= rows) u = make_uint4(0u, 0u, 0u, 0u);
    float vf[8];
    Vec8<T>::to_float(u, vf);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int v = h * NPASS + i;
      const int src = r * LPR + ((v >> (C::LOGV - C::NH)) << (C::LOGL - C::NH));
      const float pp = __shfl_sync(kFull, p[v & (NF - 1)], src);
      lsum[h] += pp;
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[h][c] = fmaf(pp, vf[c], acc[h][c]);
    }
  }
}

template <typename T, int D, int G, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32)
paged_decode_kernel(const DecodeArgs a) {
  using C = DecodeCfg<T, D, G, NW, STAGES>;
  constexpr int LPR = C::LPR;
  extern __shared__ __align__(1024) unsigned char smem[];

  const int g = blockIdx.x, s = blockIdx.y, part = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & (LPR - 1), r = lane / LPR;
  const int hq0 = g * a.group;

  int L = a.context_lens[s];
  const int max_len = a.max_blocks_per_seq * kBlock;
  if (L < 0 || L > max_len) {
    if (threadIdx.x == 0 && part == 0 && g == 0) flag(a.status, PKV_DEV_BAD_CONTEXT_LEN);
    L = L < 0 ? 0 : max_len;
  }
  const int nparts = L == 0 ? 1 : (L + a.part_tokens - 1) / a.part_tokens;
  if (part >= nparts) return;

  if (L == 0) {  // empty sequence: zeros
    T* o = static_cast<T*>(a.out) + (size_t(s) * a.num_q_heads + hq0) * D;
    for (int i = threadIdx.x; i < a.group * D / 8; i += NW * 32)
      reinterpret_cast<uint4*>(o)[i] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }

  const int t0 = part * a.part_tokens;
  const int ntok = min(L, t0 + a.part_tokens) - t0;
  const int nb = (ntok + kBlock - 1) / kBlock;

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
  int ids = load_ids(0);
  int ids_next = n_my > 32 ? load_ids(1) : 0;
  int id_batch = 0;

  const char* kbase = static_cast<const char*>(a.k_pool) + size_t(g) * C::TILE_BYTES;
  const char* vbase = static_cast<const char*>(a.v_pool) + size_t(g) * C::TILE_BYTES;
  const size_t blk_stride = size_t(a.num_kv_heads) * C::TILE_BYTES;

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
      const uint32_t bytes = uint32_t(rows) * C::ROW_BYTES;
      const int st = k % STAGES;
      const uint32_t bar = bar_s + 8 * st;
      const uint32_t dst = ring_s + st * C::STAGE_BYTES;
      mbar_arrive_expect_tx(bar, 2 * bytes);
      bulk_g2s(dst, kbase + size_t(id) * blk_stride, bytes, bar);
      bulk_g2s(dst + C::TILE_BYTES, vbase + size_t(id) * blk_stride, bytes, bar);
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
    const int j = warp + k * NW;
    const int rows = min(kBlock, ntok - j * kBlock);
    const uint32_t kt = ring_s + st * C::STAGE_BYTES;
    if (rows == kBlock)
      decode_tile<T, D, G, NW, STAGES, false>(kt, kt + C::TILE_BYTES, rows, qf, acc, lsum, mrun, lane);
    else
      decode_tile<T, D, G, NW, STAGES, true>(kt, kt + C::TILE_BYTES, rows, qf, acc, lsum, mrun, lane);
    __syncwarp();
    if (k + STAGES < n_my) issue(k + STAGES);
  }

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

  // Merge the warps: rescale each warp's sums to the common max.
  const bool direct = nparts == 1;
  constexpr int CHUNKS = D / 8;
  for (int it = threadIdx.x; it < a.group * CHUNKS; it += NW * 32) {
    const int h = it / CHUNKS, c8 = it % CHUNKS;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      M = fmaxf(M, reinterpret_cast<const float*>(smem + size_t(w) * STAGES * C::STAGE_BYTES)[G * D + h]);
    float den = 0.f, num[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) num[c] = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* ws = reinterpret_cast<const float*>(smem + size_t(w) * STAGES * C::STAGE_BYTES);
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
}

// Log-sum-exp merge of split-K partitions, one CTA (D threads) per (seq, q head):
//   M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p.
template <typename T, int D>
__global__ void __launch_bounds__(D)
paged_decode_merge_kernel(const DecodeArgs a) {
  extern __shared__ float wts[];  // [max_parts]
  __shared__ float red[D / 32];
  const int hq = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int L = a.context_lens[s];
  const int max_len = a.max_blocks_per_seq * kBlock;
  L = L < 0 ? 0 : (L > max_len ? max_len : L);
  const int nparts = L == 0 ? 1 : (L + a.part_tokens - 1) / a.part_tokens;
  if (nparts <= 1) return;  // written by the decode kernel
  const size_t row = size_t(s) * a.num_q_heads + hq;
  const float2* ml = a.part_ml + row * a.max_parts;

  float m = -INFINITY;
  for (int p = tid; p < nparts; p += D) m = fmaxf(m, ml[p].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();

  float den = 0.f;
  for (int p = tid; p < nparts; p += D) {
    const float2 x = ml[p];
    const float w = fast_exp2(x.x - M);
    wts[p] = w;
    den = fmaf(w, x.y, den);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
  if (lane == 0) red[warp] = den;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < D / 32; ++w) tot += red[w];

  const float* po = a.part_o + row * a.max_parts * D + tid;
  float acc = 0.f;
  for (int p = 0; p < nparts; ++p) acc = fmaf(wts[p], po[size_t(p) * D], acc);
  const float val = acc / tot;
  T* o = static_cast<T*>(a.out) + row * D;
  if constexpr (sizeof(T) == 2) {
    if constexpr (std::is_same<T, __half>::value)
      o[tid] = __float2half_rn(val);
    else
      o[tid] = __float2bfloat16_rn(val);
  }
}

}  // namespace pkv
