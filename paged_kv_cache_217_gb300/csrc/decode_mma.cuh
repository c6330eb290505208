// PagedAttention decode for GQA groups on the tensor cores (sm_103a).
//
// Same computation, grid, per-warp pipeline and epilogue as the CUDA-core
// kernel in decode.cuh (see its header for what is computed and the pages it
// follows). What changes is how one 16-token tile is contracted: with G >= 2
// query heads per KV head, the per-tile work is a small matrix product,
//     S[G x 16] = Q[G x D] . K^T[D x 16],   O[G x D] += P[G x 16] . V[16 x D],
// which runs as mma.sync m16n8k16 (fp16/bf16 inputs, fp32 accumulators) with
// the G heads on the M dimension (rows G..15 are zero padding). This cuts the
// issued instructions per tile by about 10x against fp32 FMAs and shuffles.
//
// Tiles arrive by TMA tensor copies (cp.async.bulk.tensor, 128-byte swizzle):
// the pool is seen as a 2-D tensor [num_blocks*num_kv_heads*16 rows, D cols]
// and each tile as D/64 boxes of 16 rows x 64 columns (a partial last tile as
// boxes of 8 and 4 rows covering its valid rows). The swizzle makes the
// ldmatrix reads of K rows (and the transposed reads of V rows) free of bank
// conflicts, which rows 256 bytes apart would otherwise hit 8 ways.
//
// P is fed to the PV product as two fp16/bf16 terms, hi = round(P) and
// lo = round(P - hi), so the weights keep about 16 significant bits instead
// of the 8 (bf16) or 11 (fp16) a single rounding leaves.
#pragma once

#include <cuda.h>

#include "decode.cuh"

namespace pkv {

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <typename T>
struct Mma;

template <>
struct Mma<__nv_bfloat16> {
  // c += a (16x16, row) . b (16x8, col), fp32 accumulate
  static __device__ __forceinline__ void run(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  // Packs two floats rounded to nearest even; returns the packed pair and
  // writes back the values it represents.
  static __device__ __forceinline__ uint32_t pack(float x, float y, float& xr, float& yr) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 f = __bfloat1622float2(h);
    xr = f.x;
    yr = f.y;
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

template <>
struct Mma<__half> {
  static __device__ __forceinline__ void run(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint32_t pack(float x, float y, float& xr, float& yr) {
    __half2 h = __floats2half2_rn(x, y);
    const float2 f = __half22float2(h);
    xr = f.x;
    yr = f.y;
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// The pool as TMA tensor maps with boxes of 16, 8 and 4 rows (index 0, 1, 2)
// x 64 columns. Full tiles are copied as 16-row boxes; a partial last tile
// with r valid rows as 4-row multiples (an 8-row box, a 4-row box, or both),
// each box landing at a 1024-byte boundary of the stage where the 128-byte
// swizzle pattern of its first row begins.
struct PoolMaps {
  CUtensorMap k[3], v[3];
};

template <typename T, int D, int NW, int STAGES>
struct MmaCfg {
  static constexpr int BOXES = D / 64;               // 64-column boxes per tile
  static constexpr int BOX_BYTES = kBlock * 128;     // 16 rows x 128 bytes
  static constexpr int TILE_BYTES = BOXES * BOX_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES; // K tile then V tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int NTILES = D / 8;
  static constexpr size_t RING_BYTES = size_t(NW) * STAGES * STAGE_BYTES;
  static constexpr size_t SMEM_BYTES = RING_BYTES + size_t(NW) * STAGES * 8 + 1024;  // + alignment slack
  static_assert(D % 64 == 0 && D >= 64 && D <= 256, "head_dim must be 64, 128 or 256");
};

// Byte offset of 16-byte chunk `chunk` (0 .. D/8-1) of row `row` (0..15) in a
// tile written by 128-byte-swizzled boxes of 16 rows x 64 columns.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return uint32_t((chunk >> 3) * (kBlock * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// One 16-row tile for the G heads of this warp's lane row g = lane/4. A lane
// whose row_on is false takes nothing from the tile (its scores are -inf):
// its weights are exactly 0 and its running max, sum and output unchanged.
template <typename T, int D, int NW, int STAGES, bool MASK>
__device__ __forceinline__ void mma_tile(uint32_t kt, uint32_t vt, int lo, int rows, const uint32_t (&qa)[D / 16][2],
                                         float (&o)[D / 8][4], float& mrun, float& lrun, float scale_log2,
                                         int lane, bool row_on = true) {
  using C = MmaCfg<T, D, NW, STAGES>;
  const int t = lane & 3;
  const int mi = lane >> 3, rr = lane & 7;

  // S = Q . K^T for tokens 0-7 (s0) and 8-15 (s1).
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int tok = (mi >> 1) * 8 + rr;
#pragma unroll
    for (int ks = 0; ks < C::KSTEPS; ++ks) {
      uint32_t b[4];
      ldsm_x4(kt + swz(tok, 2 * ks + (mi & 1)), b);
      Mma<T>::run(s0, qa[ks][0], 0u, qa[ks][1], 0u, b[0], b[1]);
      Mma<T>::run(s1, qa[ks][0], 0u, qa[ks][1], 0u, b[2], b[3]);
    }
  }

  // Online softmax on head g's scores for tokens 2t, 2t+1, 8+2t, 9+2t.
  float x[4] = {s0[0] * scale_log2, s0[1] * scale_log2, s1[0] * scale_log2, s1[1] * scale_log2};
  if (MASK) {  // only tokens [lo, rows) of the tile are valid
    if (2 * t < lo || 2 * t >= rows) x[0] = -INFINITY;
    if (2 * t + 1 < lo || 2 * t + 1 >= rows) x[1] = -INFINITY;
    if (8 + 2 * t < lo || 8 + 2 * t >= rows) x[2] = -INFINITY;
    if (9 + 2 * t < lo || 9 + 2 * t >= rows) x[3] = -INFINITY;
  }
  if (!row_on) x[0] = x[1] = x[2] = x[3] = -INFINITY;  // this lane's row (query) does not attend to this tile
  float mt = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
  mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
  const float mn = fmaxf(mrun, mt);
  // A row that has seen no valid score yet keeps mrun = -inf; exponents are
  // taken against 0 there so that every weight is exactly 0 (not NaN).
  const float mref = mn == -INFINITY ? 0.f : mn;
  if (__any_sync(kFull, mn > mrun)) {
    const float alpha = fast_exp2(mrun - mref);  // 1 for rows whose max did not move
    lrun *= alpha;
#pragma unroll
    for (int nd = 0; nd < C::NTILES; ++nd) {
      o[nd][0] *= alpha;
      o[nd][1] *= alpha;
    }
    mrun = mn;
  }
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = fast_exp2(x[i] - mref);
  lrun += (p[0] + p[1]) + (p[2] + p[3]);
  float r0, r1, r2, r3, d0, d1, d2, d3;
  const uint32_t hi01 = Mma<T>::pack(p[0], p[1], r0, r1);
  const uint32_t hi23 = Mma<T>::pack(p[2], p[3], r2, r3);
  const uint32_t lo01 = Mma<T>::pack(p[0] - r0, p[1] - r1, d0, d1);
  const uint32_t lo23 = Mma<T>::pack(p[2] - r2, p[3] - r3, d2, d3);

  // O += P . V, two n-tiles (16 dims) per transposed ldmatrix.
  {
    const int tok = (mi & 1) * 8 + rr;
#pragma unroll
    for (int c = 0; c < C::NTILES / 2; ++c) {
      uint32_t b[4];
      ldsm_x4_trans(vt + swz(tok, 2 * c + (mi >> 1)), b);
      Mma<T>::run(o[2 * c], hi01, 0u, hi23, 0u, b[0], b[1]);
      Mma<T>::run(o[2 * c], lo01, 0u, lo23, 0u, b[0], b[1]);
      Mma<T>::run(o[2 * c + 1], hi01, 0u, hi23, 0u, b[2], b[3]);
      Mma<T>::run(o[2 * c + 1], lo01, 0u, lo23, 0u, b[2], b[3]);
    }
  }
}

// Zeroes the rows outside [lo, rows) of a swizzled V tile so that 0 * (stale
// data) in the PV product cannot produce NaN, then orders these generic-proxy
// writes before the next bulk-tensor write into the same stage.
template <int D>
__device__ __forceinline__ void zero_rows_outside(uint32_t vt, int lo, int rows, int lane) {
  constexpr int CH = D / 8;
  const int n_out = lo + (kBlock - rows);
  for (int i = lane; i < n_out * CH; i += 32) {
    const int k = i / CH, chunk = i % CH;
    const int row = k < lo ? k : rows + (k - lo);
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vt + swz(row, chunk)), "r"(0u) : "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// One CTA of the shared-prefix schedule (decode_prefix.cuh, which defines it).
template <typename T, int D, int G, int NW, int STAGES>
__device__ __forceinline__ void prefix_cta(const DecodeArgs& a, const PoolMaps& maps, unsigned char* smem, int gi);

template <typename T, int D, int G, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32)
paged_decode_mma_kernel(const DecodeArgs a, const __grid_constant__ PoolMaps maps) {
  using C = MmaCfg<T, D, NW, STAGES>;
  static_assert(G >= 1 && G <= 8 && (G & (G - 1)) == 0, "tensor-core path takes groups of 1..8");
  extern __shared__ unsigned char smem_raw[];
  // 128-byte-swizzled bulk-tensor destinations want 1024-byte alignment.
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  wait_for_predecessor();
  TraceMarks tm{};
  trace_mark(tm, 0);
  const int g = blockIdx.x;
  // Shared-prefix schedule: the plan's chunks take the first grid rows
  // (longest first), the sequences outside any group the next ones; the last
  // rows (room for S chunks and S sequences, fewer used) have nothing to do.
  // Without a prefix plan of this batch the first S rows take every sequence
  // whole.
  int s;
  int4 phdr = make_int4(0, 0, 0, 0), prow0 = make_int4(-1, 0, 0, 0), prow1 = make_int4(0, 0, 0, 0);
  if (a.prefix_header) {
    const int4 ph = __ldg(a.prefix_header);
    const bool planned = ph.x == kPlanMagicPrefix && ph.y == a.num_seqs;
    const int nchunks = planned ? min(max(ph.z, 0), a.prefix_slots) : 0;
    const int nothers = planned ? min(max(ph.w, 0), a.num_seqs) : a.num_seqs;
    if (!planned && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) flag(a.status, PKV_DEV_BAD_PLAN);
    if constexpr (G == kPrefixRows) {
      if (int(blockIdx.y) < nchunks) {
        prefix_cta<T, D, G, NW, STAGES>(a, maps, smem, int(blockIdx.y));
        return;
      }
    }
    const int r = int(blockIdx.y) - nchunks;
    if (r >= nothers) return;
    s = planned ? __ldg(a.prefix_others + r) : r;
    if (s < 0 || s >= a.num_seqs) {
      if (threadIdx.x == 0 && blockIdx.x == 0) flag(a.status, PKV_DEV_BAD_PLAN);
      return;
    }
  } else {
    if (int(blockIdx.y) >= a.num_seqs) return;
    if (a.plan_rows && a.window == 0 && gridDim.z == 1) {
      phdr = __ldg(a.plan);
      prow0 = __ldg(a.plan_rows + 2 * blockIdx.y);
      prow1 = __ldg(a.plan_rows + 2 * blockIdx.y + 1);
    }
    s = long_first_seq<NW>(a, int(blockIdx.y));
  }
  const bool rows_ok = prow0.x == s && phdr.x == kPlanMagic && phdr.y == a.num_seqs;
  const int part = blockIdx.z;
  trace_mark(tm, 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq0 = g * a.group;
  const int gr = lane >> 2, t = lane & 3;   // MMA row (query head) and column pair of this lane

  // This warp's ring and barriers first: with a launch plan, the row of this
  // grid row may start the warp's first copies before its own length and
  // block ids arrive.
  unsigned char* ring = smem + size_t(warp) * STAGES * C::STAGE_BYTES;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar_s = smem_addr(smem + C::RING_BYTES) + warp * STAGES * 8;
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < STAGES; ++st) mbar_init(bar_s + 8 * st, 1);
    mbar_init_fence();
  }
  __syncwarp();

  // Lane 0 copies tile k of this warp (table position warp + k * NW of a
  // sequence stretch of ntk tokens) from physical block id.
  auto copy_tile = [&](int k, int id, int ntk) {
    if (lane == 0) {
      const int st = k % STAGES;
      const uint32_t bar = bar_s + 8 * st;
      const uint32_t dst = ring_s + st * C::STAGE_BYTES;
      const int y = (id * a.num_kv_heads + g) * kBlock;
      // rows copied: all 16, or the valid rows rounded up to a multiple of 4
      const int cover = min(kBlock, (ntk - (warp + k * NW) * kBlock + 3) & ~3);
      mbar_arrive_expect_tx(bar, uint32_t(cover) * (C::STAGE_BYTES / kBlock));
      if (cover == kBlock) {
#pragma unroll
        for (int j = 0; j < C::BOXES; ++j) {
          tma_load_2d(dst + j * C::BOX_BYTES, &maps.k[0], 64 * j, y, bar);
          tma_load_2d(dst + C::TILE_BYTES + j * C::BOX_BYTES, &maps.v[0], 64 * j, y, bar);
        }
      } else {
        // an 8-row box at row 0 when cover >= 8, then a 4-row box at row
        // (cover & 8) when cover is 4 or 12: both start on a 1024-byte boundary
#pragma unroll
        for (int j = 0; j < C::BOXES; ++j) {
          const uint32_t o = j * C::BOX_BYTES;
          if (cover & 8) {
            tma_load_2d(dst + o, &maps.k[1], 64 * j, y, bar);
            tma_load_2d(dst + C::TILE_BYTES + o, &maps.v[1], 64 * j, y, bar);
          }
          if (cover & 4) {
            const int r0 = cover & 8;
            tma_load_2d(dst + o + r0 * 128, &maps.k[2], 64 * j, y + r0, bar);
            tma_load_2d(dst + C::TILE_BYTES + o + r0 * 128, &maps.v[2], 64 * j, y + r0, bar);
          }
        }
      }
    }
  };

  // Without a sliding window the first 32 block ids of this warp's tiles do
  // not depend on the length: read them together with it (entries past the
  // sequence are never used).
  const int max_len = a.max_blocks_per_seq * kBlock;
  int ids_early = 0;
  if (a.window == 0) {
    const int j0 = (blockIdx.z * a.part_tokens) / kBlock + warp + lane * NW;
    if (j0 < a.max_blocks_per_seq) ids_early = __ldg(a.block_tables + size_t(s) * a.max_blocks_per_seq + j0);
  }
  int L = a.context_lens[s];
  // Q as the A operand: row gr holds query head hq0 + gr (zero past the group);
  // the block ids, the length and Q are all requested before the speculative
  // copies below and before anything waits for them.
  uint32_t qa[C::KSTEPS][2];
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(a.q) + (size_t(s) * a.num_q_heads + hq0 + gr) * D);
#pragma unroll
    for (int ks = 0; ks < C::KSTEPS; ++ks) {
      qa[ks][0] = gr < a.group ? __ldg(qrow + 8 * ks + t) : 0u;
      qa[ks][1] = gr < a.group ? __ldg(qrow + 8 * ks + 4 + t) : 0u;
    }
  }

  // Speculative start: the plan row's length and first block ids (table
  // positions 0..5) give this warp's first tiles. They are checked against
  // the sequence's own length and ids before the first tile is used, and
  // copied again from those if they differ (a plan made for other lengths or
  // tables), so the plan never decides a result.
  // spec: the CTA runs on the row's length (the same in every warp); spec_n:
  // the tiles this warp started from the row (0 when it has none to start).
  bool spec = false;
  int spec_n = 0, spec_len = 0;
  int spec_id[STAGES];
#pragma unroll
  for (int k = 0; k < STAGES; ++k) spec_id[k] = 0;
  if constexpr (NW * STAGES <= 6) {
    if (rows_ok && prow0.y > 0 && prow0.y <= max_len) {
      spec = true;
      spec_len = prow0.y;
      const int nb_s = (spec_len + kBlock - 1) / kBlock;
      const int n_s = min(nb_s > warp ? (nb_s - warp + NW - 1) / NW : 0, STAGES);
#pragma unroll
      for (int k = 0; k < STAGES; ++k) {
        if (k >= n_s || spec_n < k) continue;
        const int pos = warp + k * NW;
        const int id = pos == 0 ? prow0.z : pos == 1 ? prow0.w : pos == 2 ? prow1.x : pos == 3 ? prow1.y
                     : pos == 4 ? prow1.z : prow1.w;
        if (id < 0 || id >= a.num_blocks) continue;  // stop here; the sequence's own ids are checked below
        spec_id[k] = id;
        copy_tile(k, id, spec_len);
        spec_n = k + 1;
      }
    }
  }
  // Waits for the speculative copies to land (before their stages are reused or the CTA exits).
  auto drain_spec = [&]() {
#pragma unroll
    for (int k = 0; k < STAGES; ++k)
      if (k < spec_n && !mbar_wait_bounded(bar_s + 8 * k, 0) && lane == 0) flag(a.status, PKV_DEV_WAIT_TIMEOUT);
    __syncwarp();
  };

  // The sequence's length: its own (checked), or with a speculative start
  // the plan row's, compared with its own below before any tile is used.
  auto checked_len = [&](int len) {
    if (len < 0 || len > max_len) {
      if (threadIdx.x == 0 && part == 0 && g == 0) flag(a.status, PKV_DEV_BAD_CONTEXT_LEN);
      len = len < 0 ? 0 : max_len;
    }
    return len;
  };
  const int L_own = L;
  if (spec)
    L = spec_len;
  else
    L = checked_len(L_own);
  auto write_zeros = [&]() {
    T* o = static_cast<T*>(a.out) + (size_t(s) * a.num_q_heads + hq0) * D;
    for (int i = threadIdx.x; i < a.group * D / 8; i += NW * 32)
      reinterpret_cast<uint4*>(o)[i] = make_uint4(0u, 0u, 0u, 0u);
  };
  const TokenRange tr = token_range(L, a.window);
  const int nparts = L == 0 ? 1 : (L - tr.aligned + a.part_tokens - 1) / a.part_tokens;
  if (part >= nparts) return;  // (split grids only; no speculative copies there)
  const int pslot = part;  // partition slot of this CTA's partial in the workspace
  trace_mark(tm, 2);
  if (L == 0) {  // (never on the row's length)
    write_zeros();
    return;
  }
  const int t0 = tr.aligned + part * a.part_tokens;
  int ntok = min(L, t0 + a.part_tokens) - t0;
  int nb = (ntok + kBlock - 1) / kBlock;
  const int head = part == 0 ? tr.first - tr.aligned : 0;  // rows before the window in tile 0

  int n_my = nb > warp ? (nb - warp + NW - 1) / NW : 0;
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
  auto first_ids = [&]() {
    ids = 0;
    if (lane < n_my) {
      ids = a.window == 0 ? ids_early : __ldg(trow + warp + lane * NW);
      if (ids < 0 || ids >= a.num_blocks) {
        flag(a.status, PKV_DEV_BAD_BLOCK_ID);
        ids = 0;
      }
    }
  };
  int ids_next = 0, id_batch = 0;
  if (!spec) {
    first_ids();
    ids_next = n_my > 32 ? load_ids(1) : 0;
  }

  auto issue = [&](int k) {  // warp-uniform; k increases by one per call
    if ((k >> 5) != id_batch) {
      ids = ids_next;
      ++id_batch;
      ids_next = (id_batch + 1) * 32 < n_my ? load_ids(id_batch + 1) : 0;
    }
    copy_tile(k, __shfl_sync(kFull, ids, k & 31), ntok);
  };

  float o[C::NTILES][4];
#pragma unroll
  for (int nd = 0; nd < C::NTILES; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float mrun = -INFINITY, lrun = 0.f;

  // Keep the speculative copies only if they are exactly the first copies of
  // this warp (same length, same block ids); else drain them, reset the
  // barriers and copy from the sequence's own length and ids. The length
  // test is the same in every warp of the CTA.
  int pre = n_my < STAGES ? n_my : STAGES;
  bool started = false;
  if (spec) {  // (one pass, no window: ids_early holds table positions warp + lane * NW)
    const int own = checked_len(L_own);
    bool same = own == spec_len && spec_n == pre;
#pragma unroll
    for (int k = 0; k < STAGES; ++k)
      if (k < spec_n) same = same && __shfl_sync(kFull, ids_early, k) == spec_id[k];
    if (same) {
      started = true;
    } else {
      drain_spec();
      if (lane == 0) {
#pragma unroll
        for (int st = 0; st < STAGES; ++st) {
          mbar_inval(bar_s + 8 * st);
          mbar_init(bar_s + 8 * st, 1);
        }
        mbar_init_fence();
      }
      __syncwarp();
      if (own != spec_len) {  // one pass, no window: the stretch is the whole sequence
        if (own == 0) {  // every warp of the CTA comes here
          write_zeros();
          return;
        }
        L = own;
        ntok = L;
        nb = (ntok + kBlock - 1) / kBlock;
        n_my = nb > warp ? (nb - warp + NW - 1) / NW : 0;
        pre = n_my < STAGES ? n_my : STAGES;
      }
    }
    first_ids();  // checked (and flagged) against the settled tile count only
    ids_next = n_my > 32 ? load_ids(1) : 0;
  }
  if (!started)
    for (int k = 0; k < pre; ++k) issue(k);

  for (int k = 0; k < n_my; ++k) {
    const int st = k % STAGES;
    const uint32_t parity = (k / STAGES) & 1;
    const bool ok = mbar_wait_bounded(bar_s + 8 * st, parity);
    if (!__all_sync(kFull, ok)) {
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
    if (rows == kBlock && lo == 0) {
      mma_tile<T, D, NW, STAGES, false>(kt, kt + C::TILE_BYTES, 0, rows, qa, o, mrun, lrun, a.scale_log2, lane);
    } else {
      zero_rows_outside<D>(kt + C::TILE_BYTES, lo, rows, lane);
      mma_tile<T, D, NW, STAGES, true>(kt, kt + C::TILE_BYTES, lo, rows, qa, o, mrun, lrun, a.scale_log2, lane);
    }
    __syncwarp();
    if (k + STAGES < n_my) issue(k + STAGES);
  }

  trace_mark(tm, 4);
  // Row sums: the four lanes of a row each summed a quarter of the tokens.
  lrun += __shfl_xor_sync(kFull, lrun, 1);
  lrun += __shfl_xor_sync(kFull, lrun, 2);

  // Publish (acc[G][D], m[G], l[G]) in this warp's ring for the shared epilogue.
  float* wsm = reinterpret_cast<float*>(ring);
  if (gr < G) {
#pragma unroll
    for (int nd = 0; nd < C::NTILES; ++nd)
      *reinterpret_cast<float2*>(wsm + gr * D + 8 * nd + 2 * t) = make_float2(o[nd][0], o[nd][1]);
    if (t == 0) {
      wsm[G * D + gr] = mrun;
      wsm[G * D + G + gr] = lrun;
    }
  }
  __syncthreads();
  finish_chunk<T, D, G, NW>(a, smem, size_t(STAGES) * C::STAGE_BYTES, s, g, pslot, nparts);
  trace_write(a, tm, s, nb);
}

}  // namespace pkv
