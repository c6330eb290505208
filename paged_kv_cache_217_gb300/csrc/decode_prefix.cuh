// PagedAttention decode over a prompt prefix that sibling sequences share
// (sm_103a).
//
// Parallel samples of one prompt share the prompt's full blocks through
// their block tables -- the same physical blocks, reference-counted, copied
// only when a write reaches one (abeam.tech summary of "Efficient Memory
// Management for Large Language Model Serving with PagedAttention",
// "並列サンプリングやビームサーチでの共有"; glossary entry
// "PagedAttention（ページドアテンション）", "コピーオンライト（Copy-on-Write）
// 共有"). Attention is still computed per sequence exactly as in decode.cuh;
// only its work is arranged so that each shared tile is read once:
//
//  * The step's plan (prefix_plan_kernel) finds groups of consecutive
//    sequences whose tables start with the same physical blocks (P shared
//    whole blocks), and splits each group's work into 1..kPrefixMaxParts
//    chunks -- ranges of block indices -- when the batch has too few groups
//    to fill the GPU.
//  * One CTA per (KV head, chunk) (prefix_cta, run by the first CTA rows of
//    the tensor-core grid kernel): the members' query rows of the KV head
//    (members x query heads per KV head, at most 8) form the M rows of the
//    tensor-core tile (mma_tile), so each shared K/V tile is copied into
//    shared memory once and multiplied with every sibling's queries; the
//    members' own tiles in the chunk follow, each masked out of the other
//    members' rows. A group of one chunk writes its outputs directly; the
//    chunks of a split group leave partials that the last to finish merges
//    by log-sum-exp. The chunk CTAs come first in the grid, longest first;
//    the grid's later rows take the sequences outside any group.
#pragma once

#include "decode_mma.cuh"

namespace pkv {

// The chunk a shared-prefix CTA works on (chunk ci of a valid prefix plan,
// KV head blockIdx.x), and this warp's share of its tiles.
//
// The chunk covers block indices [jb, je) of its group: the shared blocks
// among them (read through the first member's table) and each member's own
// blocks among them (read through its own table). A warp takes a run of the
// shared blocks, then each member's own blocks j = warp (mod NW) in order. A
// member's row attends to the shared tiles and to its own; other members'
// tiles are masked out of it (they change nothing in that row). Siblings of
// one group with equal lengths and contents therefore get bit-identical
// outputs.
template <int NW>
struct PrefixChunk {
  int s0, members, P, parts, part, rows;
  // per member m: (length << 9) | this warp's own tiles (length <= 4096, own <= 256)
  int mem[kPrefixRows];
  int sh_first, sh_n, j_own, n_my;

  // Reads and checks the chunk; false (after flagging PKV_DEV_BAD_PLAN) when
  // the plan is not one this batch can run.
  __device__ __forceinline__ bool init(const DecodeArgs& a, int ci, int warp) {
    const int g = blockIdx.x;
    const int4 ch = __ldg(a.prefix_chunks + ci);
    const int gi = ch.x, jb = ch.z, je = ch.w;
    part = ch.y;
    const int max_groups = a.num_seqs / 2 > 0 ? a.num_seqs / 2 : 1;
    int4 grp = make_int4(-1, 0, 0, 0);
    if (gi >= 0 && gi < max_groups) grp = __ldg(a.prefix_groups + gi);
    s0 = grp.x, members = grp.y, P = grp.z, parts = grp.w;
    rows = members * a.group;
    if (gi < 0 || gi >= max_groups || s0 < 0 || members < 2 || s0 + members > a.num_seqs || rows > kPrefixRows ||
        P < kPrefixMinBlocks || P > a.max_blocks_per_seq || parts < 1 || parts > kPrefixMaxParts || part < 0 ||
        part >= parts || jb < 0 || je < jb || je > a.max_blocks_per_seq) {
      if (threadIdx.x == 0 && g == 0) flag(a.status, PKV_DEV_BAD_PLAN);
      return false;
    }
    const int max_len = a.max_blocks_per_seq * kBlock;
    // Members' lengths and own tiles per warp: a member's own blocks j go to
    // warp j mod NW (the same for every member, so equal siblings see equal
    // tiles in equal warps); the shared blocks of the chunk are cut into NW
    // consecutive runs that even out the warps' totals (water-filling over
    // the own counts).
    auto count_below = [&](int x, int w) { return x > w ? (x - w + NW - 1) / NW : 0; };  // j < x, j = w (mod NW)
    int own_w[NW];
#pragma unroll
    for (int w = 0; w < NW; ++w) own_w[w] = 0;
    const int sh_end = min(je, P), own_lo = max(jb, P);
    const int sh_total = jb < sh_end ? sh_end - jb : 0;
#pragma unroll
    for (int m = 0; m < kPrefixRows; ++m) {
      int L = m < members ? __ldg(a.context_lens + s0 + m) : 0;
      L = L < 0 ? 0 : (L > max_len ? max_len : L);
      if (m < members && L < P * kBlock) {  // the plan promised P whole blocks of every member
        if (threadIdx.x == 0 && g == 0) flag(a.status, PKV_DEV_BAD_PLAN);
        L = P * kBlock;
      }
      const int hi = min(je, (L + kBlock - 1) / kBlock);
      int mine = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const int c = (m < members && own_lo < hi) ? count_below(hi, w) - count_below(own_lo, w) : 0;
        own_w[w] += c;
        if (w == warp) mine = c;
      }
      mem[m] = (L << 9) | mine;
    }
    // the smallest level L with sum_w max(0, L - own_w) >= sh_total; warps
    // below L - 1 fill up to it, the first few at L - 1 take the remainder
    int lo = 0, hi = sh_total;
#pragma unroll
    for (int w = 0; w < NW; ++w) hi = max(hi, own_w[w] + sh_total);
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      int fill = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) fill += max(0, mid - own_w[w]);
      if (fill >= sh_total) hi = mid; else lo = mid + 1;
    }
    int rest = sh_total;
#pragma unroll
    for (int w = 0; w < NW; ++w) rest -= max(0, lo - 1 - own_w[w]);
    sh_n = 0;
    sh_first = jb;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      int n = max(0, lo - 1 - own_w[w]);
      if (rest > 0 && own_w[w] <= lo - 1) {
        ++n;
        --rest;
      }
      if (w < warp) sh_first += n;
      if (w == warp) sh_n = n;
    }
    n_my = sh_n;
#pragma unroll
    for (int m = 0; m < kPrefixRows; ++m) n_my += mem[m] & 511;
    j_own = own_lo + ((warp - own_lo) % NW + NW) % NW;  // the first own block j >= own_lo of this warp
    return true;
  }

  // Tile k of this warp: (member, block, valid rows) -- member -1 for a
  // shared tile. (The arrays are indexed with unrolled constants only, so
  // they stay in registers.)
  __device__ __forceinline__ void locate(int k, int& m, int& j, int& rows) const {
    m = -1;
    j = sh_first + k;
    rows = kBlock;
    if (k < sh_n) return;
    int r = k - sh_n;
#pragma unroll
    for (int mm = 0; mm < kPrefixRows; ++mm) {
      const int own = mem[mm] & 511;
      if (m < 0 && r < own) {
        m = mm;
        j = j_own + r * NW;
        rows = min(kBlock, (mem[mm] >> 9) - j * kBlock);
      }
      if (m < 0) r -= own;
    }
  }
  // Physical block of tile (m, j), checked against the pool (0 and flagged if bad).
  __device__ __forceinline__ int block_id(const DecodeArgs& a, int m, int j) const {
    int id = __ldg(a.block_tables + size_t(s0 + (m < 0 ? 0 : m)) * a.max_blocks_per_seq + j);
    if (id < 0 || id >= a.num_blocks) {
      flag(a.status, PKV_DEV_BAD_BLOCK_ID);
      id = 0;
    }
    return id;
  }
};

// The end of a shared-prefix CTA: every warp has published (acc[G][D], m[G],
// l[G]) at the start of its ring (acc unnormalised, in head-dim order) and
// the CTA has synchronised. Merges the warps per row; a group of one chunk
// writes its outputs, a chunk of a split group leaves its partial (a row
// without tiles in the chunk leaves M = -inf), and the last chunk of the
// group to finish (for this KV head) merges the parts by log-sum-exp.
template <typename T, int D, int G, int NW>
__device__ __forceinline__ void prefix_finish(const DecodeArgs& a, const PrefixChunk<NW>& c,
                                              const unsigned char* smem, size_t area) {
  constexpr int CHUNKS = D / 8;
  const int g = blockIdx.x;
  for (int it = threadIdx.x; it < c.rows * CHUNKS; it += NW * 32) {
    const int r = it / CHUNKS, c8 = it % CHUNKS;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<const float*>(smem + size_t(w) * area)[G * D + r]);
    float den = 0.f, num[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) num[k] = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* ws = reinterpret_cast<const float*>(smem + size_t(w) * area);
      const float mw = ws[G * D + r];
      if (mw == -INFINITY) continue;
      const float wt = fast_exp2(mw - M);
      den = fmaf(wt, ws[G * D + G + r], den);
      const float4* src = reinterpret_cast<const float4*>(ws + r * D + c8 * 8);
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
    const size_t row = size_t(c.s0 + r / a.group) * a.num_q_heads + g * a.group + r % a.group;
    if (c.parts == 1) {  // every row has seen its shared tiles: den > 0
      const float inv = 1.f / den;
#pragma unroll
      for (int k = 0; k < 8; ++k) num[k] *= inv;
      reinterpret_cast<uint4*>(static_cast<T*>(a.out) + row * D)[c8] = Vec8<T>::from_float(num);
    } else {
      float4* dst = reinterpret_cast<float4*>(a.part_o + (row * kPrefixMaxParts + c.part) * D + c8 * 8);
      dst[0] = make_float4(num[0], num[1], num[2], num[3]);
      dst[1] = make_float4(num[4], num[5], num[6], num[7]);
      if (c8 == 0) a.part_ml[row * kPrefixMaxParts + c.part] = make_float2(M, den);
    }
  }
  if (c.parts == 1) return;

  __shared__ unsigned int prefix_last;
  __threadfence();
  __syncthreads();
  unsigned int* counter = a.counters + size_t(c.s0) * a.num_kv_heads + g;
  if (threadIdx.x == 0) prefix_last = atomicAdd(counter, 1u) == unsigned(c.parts - 1) ? 1u : 0u;
  __syncthreads();
  if (!prefix_last) return;
  __threadfence();
  for (int it = threadIdx.x; it < c.rows * CHUNKS; it += NW * 32) {
    const int r = it / CHUNKS, c8 = it % CHUNKS;
    const size_t row = size_t(c.s0 + r / a.group) * a.num_q_heads + g * a.group + r % a.group;
    const float2* ml = a.part_ml + row * kPrefixMaxParts;
    const float* po = a.part_o + row * kPrefixMaxParts * D + c8 * 8;
    float M = -INFINITY;
    for (int p = 0; p < c.parts; ++p) M = fmaxf(M, __ldcg(&ml[p].x));
    float den = 0.f, num[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) num[k] = 0.f;
    for (int p = 0; p < c.parts; ++p) {
      const float2 x = __ldcg(ml + p);
      if (x.x == -INFINITY) continue;  // no tile of this row in that chunk
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
    for (int k = 0; k < 8; ++k) num[k] *= inv;
    reinterpret_cast<uint4*>(static_cast<T*>(a.out) + row * D)[c8] = Vec8<T>::from_float(num);
  }
  if (threadIdx.x == 0) *counter = 0u;  // leave the workspace ready for the next call
}

// One CTA of the shared-prefix schedule on the 16-bit cache. Called by the
// tensor-core grid kernel; `smem` is that kernel's 1024-byte-aligned shared
// memory (rings of NW warps x STAGES stages).
template <typename T, int D, int G, int NW, int STAGES>
__device__ __forceinline__ void prefix_cta(const DecodeArgs& a, const PoolMaps& maps, unsigned char* smem, int ci) {
  using C = MmaCfg<T, D, NW, STAGES>;
  static_assert(G == kPrefixRows, "a group's rows fill the tile's G rows");

  const int g = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;  // MMA row and column pair of this lane
  PrefixChunk<NW> c;
  if (!c.init(a, ci, warp)) return;

  unsigned char* ring = smem + size_t(warp) * STAGES * C::STAGE_BYTES;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar_s = smem_addr(smem + C::RING_BYTES) + warp * STAGES * 8;
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < STAGES; ++st) mbar_init(bar_s + 8 * st, 1);
    mbar_init_fence();
  }
  __syncwarp();

  // The A operand: row r is query head g * group + r % group of member r / group.
  uint32_t qa[C::KSTEPS][2];
  const int my_member = gr / a.group;
  {
    const int h = g * a.group + gr % a.group;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(a.q) + (size_t(c.s0 + (gr < c.rows ? my_member : 0)) * a.num_q_heads + h) * D);
#pragma unroll
    for (int ks = 0; ks < C::KSTEPS; ++ks) {
      qa[ks][0] = gr < c.rows ? __ldg(qrow + 8 * ks + t) : 0u;
      qa[ks][1] = gr < c.rows ? __ldg(qrow + 8 * ks + 4 + t) : 0u;
    }
  }

  // lane l of a batch holds the block id of this warp's tile k = batch * 32 + l
  const int n_my = c.n_my;
  auto load_ids = [&](int batch) -> int {
    const int k = batch * 32 + lane;
    if (k >= n_my) return 0;
    int m, j, rows;
    c.locate(k, m, j, rows);
    return c.block_id(a, m, j);
  };
  int ids = load_ids(0);
  int ids_next = n_my > 32 ? load_ids(1) : 0;
  int id_batch = 0;
  auto issue = [&](int k) {  // warp-uniform; k increases by one per call
    if ((k >> 5) != id_batch) {
      ids = ids_next;
      ++id_batch;
      ids_next = (id_batch + 1) * 32 < n_my ? load_ids(id_batch + 1) : 0;
    }
    const int id = __shfl_sync(kFull, ids, k & 31);
    if (lane == 0) {
      int m, j, rows;
      c.locate(k, m, j, rows);
      const int cover = min(kBlock, (rows + 3) & ~3);  // rows copied, a multiple of 4
      const int st = k % STAGES;
      const uint32_t bar = bar_s + 8 * st;
      const uint32_t dst = ring_s + st * C::STAGE_BYTES;
      const int y = (id * a.num_kv_heads + g) * kBlock;
      mbar_arrive_expect_tx(bar, uint32_t(cover) * (C::STAGE_BYTES / kBlock));
      if (cover == kBlock) {
#pragma unroll
        for (int jb2 = 0; jb2 < C::BOXES; ++jb2) {
          tma_load_2d(dst + jb2 * C::BOX_BYTES, &maps.k[0], 64 * jb2, y, bar);
          tma_load_2d(dst + C::TILE_BYTES + jb2 * C::BOX_BYTES, &maps.v[0], 64 * jb2, y, bar);
        }
      } else {
#pragma unroll
        for (int jb2 = 0; jb2 < C::BOXES; ++jb2) {
          const uint32_t o = jb2 * C::BOX_BYTES;
          if (cover & 8) {
            tma_load_2d(dst + o, &maps.k[1], 64 * jb2, y, bar);
            tma_load_2d(dst + C::TILE_BYTES + o, &maps.v[1], 64 * jb2, y, bar);
          }
          if (cover & 4) {
            const int r0 = cover & 8;
            tma_load_2d(dst + o + r0 * 128, &maps.k[2], 64 * jb2, y + r0, bar);
            tma_load_2d(dst + C::TILE_BYTES + o + r0 * 128, &maps.v[2], 64 * jb2, y + r0, bar);
          }
        }
      }
    }
  };

  float o[C::NTILES][4];
#pragma unroll
  for (int nd = 0; nd < C::NTILES; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float mrun = -INFINITY, lrun = 0.f;
  const int pre = n_my < STAGES ? n_my : STAGES;
  for (int k = 0; k < pre; ++k) issue(k);
  for (int k = 0; k < n_my; ++k) {
    const int st = k % STAGES;
    const bool ok = mbar_wait_bounded(bar_s + 8 * st, (k / STAGES) & 1);
    if (!__all_sync(kFull, ok)) {
      if (lane == 0) flag(a.status, PKV_DEV_WAIT_TIMEOUT);
      const int last = min(n_my, k + STAGES);
      for (int kk = k; kk < last; ++kk) mbar_wait_bounded(bar_s + 8 * (kk % STAGES), (kk / STAGES) & 1);
      break;
    }
    int m, j, valid;
    c.locate(k, m, j, valid);
    const bool row_on = m < 0 || my_member == m;
    const uint32_t kt = ring_s + st * C::STAGE_BYTES;
    if (valid == kBlock) {
      mma_tile<T, D, NW, STAGES, false>(kt, kt + C::TILE_BYTES, 0, kBlock, qa, o, mrun, lrun, a.scale_log2, lane,
                                        row_on);
    } else {
      zero_rows_outside<D>(kt + C::TILE_BYTES, 0, valid, lane);
      mma_tile<T, D, NW, STAGES, true>(kt, kt + C::TILE_BYTES, 0, valid, qa, o, mrun, lrun, a.scale_log2, lane,
                                       row_on);
    }
    __syncwarp();
    if (k + STAGES < n_my) issue(k + STAGES);
  }
  lrun += __shfl_xor_sync(kFull, lrun, 1);
  lrun += __shfl_xor_sync(kFull, lrun, 2);

  // Publish (acc[G][D], m[G], l[G]) in this warp's ring, as the grid kernels do.
  float* wsm = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int nd = 0; nd < C::NTILES; ++nd)
    *reinterpret_cast<float2*>(wsm + gr * D + 8 * nd + 2 * t) = make_float2(o[nd][0], o[nd][1]);
  if (t == 0) {
    wsm[G * D + gr] = mrun;
    wsm[G * D + G + gr] = lrun;
  }
  __syncthreads();
  prefix_finish<T, D, G, NW>(a, c, smem, size_t(STAGES) * C::STAGE_BYTES);
}

}  // namespace pkv
