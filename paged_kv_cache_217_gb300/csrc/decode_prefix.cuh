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
//    sequences whose tables start with the same physical blocks, and for each
//    member the number of shared tokens (whole blocks, at most every member's
//    length rounded down to a block).
//  * One CTA per (KV head, group) (prefix_cta, run by the first CTA rows of
//    the tensor-core grid kernel): the members' query rows
//    of the KV head (members x query heads per KV head, at most 8) form the M
//    rows of the tensor-core tile (mma_tile), so each shared K/V tile is
//    copied into shared memory once and multiplied with every sibling's
//    queries. Its result per row is a partial (max, sum, unnormalised V sum)
//    over the shared tokens, in workspace slot 0 of that row.
//  * The grid's other CTAs take each member's remaining tokens (slot 1); the
//    last of the two to finish (an arrival counter per sequence and KV head)
//    merges them by log-sum-exp. A member without tokens of its own gets its
//    output straight from its group's CTA. The group CTAs come first in the
//    grid (they are the long ones), so the members' short CTAs fill the GPU
//    around them.
#pragma once

#include "decode_mma.cuh"

namespace pkv {

// One CTA of the shared-prefix schedule: the group of blockIdx.y (a slot of
// the plan's group list; past the list, nothing), KV head blockIdx.x. Called
// by the tensor-core grid kernel, whose CTAs past the group slots take the
// members' own tokens; `smem` is that kernel's 1024-byte-aligned shared
// memory (rings of NW warps x STAGES stages).
template <typename T, int D, int G, int NW, int STAGES>
__device__ __forceinline__ void prefix_cta(const DecodeArgs& a, const PoolMaps& maps, unsigned char* smem, int gi) {
  using C = MmaCfg<T, D, NW, STAGES>;
  static_assert(G == kPrefixRows, "a group's rows fill the tile's G rows");
  constexpr int CHUNKS = D / 8;

  const int g = blockIdx.x;
  const int4 hdr = __ldg(a.prefix_header);
  if (hdr.x != kPlanMagicPrefix || hdr.y != a.num_seqs) {  // no plan: the sequences' CTAs do everything
    if (threadIdx.x == 0 && g == 0 && gi == 0) flag(a.status, PKV_DEV_BAD_PLAN);
    return;
  }
  if (gi >= hdr.z) return;
  const int4 grp = __ldg(a.prefix_groups + gi);
  const int s0 = grp.x, members = grp.y, P = grp.z;
  const int rows = members * a.group;
  if (s0 < 0 || members < 2 || s0 + members > a.num_seqs || rows > G || P < 1 || P > a.max_blocks_per_seq) {
    if (threadIdx.x == 0 && g == 0) flag(a.status, PKV_DEV_BAD_PLAN);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;  // MMA row and column pair of this lane

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
  {
    const int m = gr / a.group, h = g * a.group + gr % a.group;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(a.q) + (size_t(s0 + (gr < rows ? m : 0)) * a.num_q_heads + h) * D);
#pragma unroll
    for (int ks = 0; ks < C::KSTEPS; ++ks) {
      qa[ks][0] = gr < rows ? __ldg(qrow + 8 * ks + t) : 0u;
      qa[ks][1] = gr < rows ? __ldg(qrow + 8 * ks + 4 + t) : 0u;
    }
  }

  // Tiles j = warp, warp + NW, ... of the shared blocks, read through the
  // first member's table (every member's table holds the same ids there).
  const int n_my = P > warp ? (P - warp + NW - 1) / NW : 0;
  const int32_t* trow = a.block_tables + size_t(s0) * a.max_blocks_per_seq;
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
  auto issue = [&](int k) {  // warp-uniform; k increases by one per call; every tile is full
    if ((k >> 5) != id_batch) {
      ids = ids_next;
      ++id_batch;
      ids_next = (id_batch + 1) * 32 < n_my ? load_ids(id_batch + 1) : 0;
    }
    const int id = __shfl_sync(kFull, ids, k & 31);
    if (lane == 0) {
      const int st = k % STAGES;
      const uint32_t bar = bar_s + 8 * st;
      const uint32_t dst = ring_s + st * C::STAGE_BYTES;
      const int y = (id * a.num_kv_heads + g) * kBlock;
      mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
#pragma unroll
      for (int j = 0; j < C::BOXES; ++j) {
        tma_load_2d(dst + j * C::BOX_BYTES, &maps.k[0], 64 * j, y, bar);
        tma_load_2d(dst + C::TILE_BYTES + j * C::BOX_BYTES, &maps.v[0], 64 * j, y, bar);
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
    const uint32_t kt = ring_s + st * C::STAGE_BYTES;
    mma_tile<T, D, NW, STAGES, false>(kt, kt + C::TILE_BYTES, 0, kBlock, qa, o, mrun, lrun, a.scale_log2, lane);
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

  // Merge the warps; each row's result is its member's output (no own
  // tokens) or the member's partial in slot 0.
  const int max_len = a.max_blocks_per_seq * kBlock;
  const size_t area = size_t(STAGES) * C::STAGE_BYTES;
  for (int it = threadIdx.x; it < rows * CHUNKS; it += NW * 32) {
    const int r = it / CHUNKS, c8 = it % CHUNKS;
    const int s = s0 + r / a.group, hq = g * a.group + r % a.group;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<const float*>(smem + size_t(w) * area)[G * D + r]);
    float den = 0.f, num[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) num[c] = 0.f;
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
    int L = __ldg(a.context_lens + s);
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    const size_t row = size_t(s) * a.num_q_heads + hq;
    if (L <= P * kBlock) {  // the shared tokens are all of this member's tokens
      const float inv = 1.f / den;
#pragma unroll
      for (int c = 0; c < 8; ++c) num[c] *= inv;
      reinterpret_cast<uint4*>(static_cast<T*>(a.out) + row * D)[c8] = Vec8<T>::from_float(num);
    } else {
      float4* dst = reinterpret_cast<float4*>(a.part_o + (row * a.max_parts + 0) * D + c8 * 8);
      dst[0] = make_float4(num[0], num[1], num[2], num[3]);
      dst[1] = make_float4(num[4], num[5], num[6], num[7]);
      if (c8 == 0) a.part_ml[row * a.max_parts + 0] = make_float2(M, den);
    }
  }

  // One arrival per member with tokens of its own; the last of the two
  // partitions of a (sequence, KV head) merges them.
  __shared__ int last_m[kPrefixRows];
  __threadfence();
  __syncthreads();
  if (threadIdx.x < members) {
    const int s = s0 + threadIdx.x;
    int L = __ldg(a.context_lens + s);
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    last_m[threadIdx.x] = 0;
    if (L > P * kBlock)
      last_m[threadIdx.x] = atomicAdd(a.counters + size_t(s) * a.num_kv_heads + g, 1u) == 1u ? 1 : 0;
  }
  __syncthreads();
  __threadfence();
  for (int it = threadIdx.x; it < rows * CHUNKS; it += NW * 32) {
    const int r = it / CHUNKS, c8 = it % CHUNKS;
    if (!last_m[r / a.group]) continue;
    const int s = s0 + r / a.group, hq = g * a.group + r % a.group;
    const size_t row = size_t(s) * a.num_q_heads + hq;
    const float2* ml = a.part_ml + row * a.max_parts;
    const float* po = a.part_o + row * a.max_parts * D + c8 * 8;
    float M = -INFINITY;
    for (int q = 0; q < 2; ++q) M = fmaxf(M, __ldcg(&ml[q].x));
    float den = 0.f, num[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) num[c] = 0.f;
    for (int q = 0; q < 2; ++q) {
      const float2 x = __ldcg(ml + q);
      const float w = fast_exp2(x.x - M);
      den = fmaf(w, x.y, den);
      const float4* src = reinterpret_cast<const float4*>(po + size_t(q) * D);
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
  __syncthreads();
  if (threadIdx.x < members && last_m[threadIdx.x])
    a.counters[size_t(s0 + threadIdx.x) * a.num_kv_heads + g] = 0u;  // ready for the next call
}

}  // namespace pkv
