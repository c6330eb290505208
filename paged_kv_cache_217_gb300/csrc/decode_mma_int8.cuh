// PagedAttention decode over the INT8 KV cache on the tensor cores (sm_103a).
//
// Computes what the CUDA-core INT8 path computes (decode.cuh with KvInt8):
// attention over K = c_K * s_K and V = c_V * s_V, one fp32 scale per stored
// row. The INT8 cache is the companion of paging named by the glossary entry
// "PagedAttention（ページドアテンション）" (section
// "他のKVキャッシュ最適化との組み合わせ").
//
// Per 16-token tile, as mma.sync m16n8k16 with fp16 inputs and fp32
// accumulators (query heads on M, rows G..15 zero):
//  * S = Q~ . C_K^T. Codes become fp16 exactly in registers: a byte b, biased
//    to b + 128, is placed under the exponent byte 0x64 (fp16 1024 + b + 128)
//    and 1152 is subtracted. Q~ is q times a power of two per head (bringing
//    max|q| to [2^13, 2^14), so bf16 queries are exact in fp16); the fp32
//    scores are then multiplied by s_K of their token, the inverse power of
//    two and scale * log2(e).
//    The contraction runs over a permuted order of the head dims: k-slots
//    2t, 2t+1, 2t+8, 2t+9 of a 16-dim chunk hold dims 4t .. 4t+3, so each
//    K fragment is one 32-bit shared-memory word.
//  * O += P . V~ with V~ = c_V * s_V rounded to fp16 (the exact code pair
//    times the fp16 pair of scales), P rounded to fp16 once. Each
//    lane loads one 32-bit word (4 dims) from each of its 4 token rows and
//    regroups the bytes so that output column slot s of n-tile 4g + i holds
//    head dim 32g + 4s + i; the epilogue undoes that permutation.
//  * K and V tiles arrive by TMA tensor copies of uint8 boxes (16 rows x
//    min(D, 128) bytes) with the 128-byte swizzle (64-byte at D = 64), which
//    keeps the word loads above free of bank conflicts; the 16 K and 16 V
//    scales of the tile arrive by two 64-byte bulk copies.
// Rounding V~ and P to fp16 each adds at most 2^-12 relative error per term,
// far below the quantisation step of the codes.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "decode_mma.cuh"

namespace pkv {

template <int D, int NW, int STAGES>
struct I8Cfg {
  static constexpr int BOX_COLS = D < 128 ? D : 128;  // bytes per box row
  static constexpr int BOXES = D / BOX_COLS;
  static constexpr int BOX_BYTES = kBlock * BOX_COLS;
  static constexpr int TILE_BYTES = kBlock * D;       // one K (or V) tile of codes
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
  static constexpr int SCALE_STAGE = 2 * kBlock * 4;  // 16 K scales then 16 V scales
  static constexpr int KCHUNKS = D / 16;              // QK k-steps
  static constexpr int VGROUPS = D / 32;              // PV groups of 4 n-tiles
  static constexpr int NTILES = D / 8;
  static constexpr size_t RING_BYTES = size_t(NW) * STAGES * STAGE_BYTES;
  static constexpr size_t SCALE_BYTES = size_t(NW) * STAGES * SCALE_STAGE;
  static constexpr size_t SMEM_BYTES = RING_BYTES + SCALE_BYTES + size_t(NW) * STAGES * 8 + 1024;
  static_assert(D == 64 || D == 128 || D == 256, "head_dim must be 64, 128 or 256");
  static_assert(size_t(8 * 2 + 8 * D) * 4 <= size_t(STAGES) * STAGE_BYTES, "merge area fits the ring");
};

// Byte offset of 16-byte chunk `ch` of row `row` in a swizzled code tile.
template <int D>
__device__ __forceinline__ uint32_t i8_swz(int row, int ch) {
  if constexpr (D == 64) {
    return uint32_t(row * 64 + (((ch & 3) ^ ((row >> 1) & 3)) << 4));
  } else {
    return uint32_t((ch >> 3) * (kBlock * 128) + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
  }
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ float2 lds_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

constexpr uint32_t kF16Magic = 0x64646464u;   // fp16 exponent byte of 1024
constexpr uint32_t kF16Bias = 0x64806480u;    // fp16x2 (1152, 1152)

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Four int8 codes (one word) -> two fp16x2 registers: bytes (0, 1) and (2, 3), exact.
__device__ __forceinline__ void codes_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  lo = hsub2_u32(__byte_perm(x, kF16Magic, 0x5140), kF16Bias);
  hi = hsub2_u32(__byte_perm(x, kF16Magic, 0x5342), kF16Bias);
}

template <int D, int NW, int STAGES, bool MASK>
__device__ __forceinline__ void mma_tile_int8(uint32_t kt, uint32_t vt, uint32_t st_scale, int lo, int rows,
                                              const uint32_t (&qa)[D / 16][2], float (&o)[D / 8][4],
                                              float& mrun, float& lrun, float qmul, int lane) {
  using C = I8Cfg<D, NW, STAGES>;
  const int t = lane & 3, gr = lane >> 2;

  // S = Q~ . C_K^T: n-tile 0 = tokens 0..7 (this lane's token gr), n-tile 1 = tokens 8..15.
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < C::KCHUNKS; ++c) {
    const uint32_t w0 = lds32(kt + i8_swz<D>(gr, c) + 4 * t);
    const uint32_t w1 = lds32(kt + i8_swz<D>(gr + 8, c) + 4 * t);
    uint32_t b0, b1, b2, b3;
    codes_to_f16x2(w0, b0, b1);
    codes_to_f16x2(w1, b2, b3);
    Mma<__half>::run(s0, qa[c][0], 0u, qa[c][1], 0u, b0, b1);
    Mma<__half>::run(s1, qa[c][0], 0u, qa[c][1], 0u, b2, b3);
  }

  // Scores of head gr for tokens 2t, 2t+1, 8+2t, 9+2t, in the log2 domain.
  const float2 ka = lds_f32x2(st_scale + 8 * t);
  const float2 kb = lds_f32x2(st_scale + 32 + 8 * t);
  float x[4] = {s0[0] * ka.x * qmul, s0[1] * ka.y * qmul, s1[0] * kb.x * qmul, s1[1] * kb.y * qmul};
  if (MASK) {
    if (2 * t < lo || 2 * t >= rows) x[0] = -INFINITY;
    if (2 * t + 1 < lo || 2 * t + 1 >= rows) x[1] = -INFINITY;
    if (8 + 2 * t < lo || 8 + 2 * t >= rows) x[2] = -INFINITY;
    if (9 + 2 * t < lo || 9 + 2 * t >= rows) x[3] = -INFINITY;
  }
  float mt = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
  mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
  const float mn = fmaxf(mrun, mt);
  if (__any_sync(kFull, mn > mrun)) {
    const float alpha = fast_exp2(mrun - mn);
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
  for (int i = 0; i < 4; ++i) p[i] = fast_exp2(x[i] - mn);
  lrun += (p[0] + p[1]) + (p[2] + p[3]);
  const __half2 p01 = __floats2half2_rn(p[0], p[1]);
  const __half2 p23 = __floats2half2_rn(p[2], p[3]);
  const uint32_t a01 = *reinterpret_cast<const uint32_t*>(&p01);
  const uint32_t a23 = *reinterpret_cast<const uint32_t*>(&p23);

  // V scales of tokens (2t, 2t+1) and (2t+8, 2t+9) as fp16 pairs; rows outside
  // [lo, rows) get scale 0 so their (stale) codes contribute exactly nothing.
  const float2 va = lds_f32x2(st_scale + 64 + 8 * t);
  const float2 vb = lds_f32x2(st_scale + 96 + 8 * t);
  float sv[4] = {va.x, va.y, vb.x, vb.y};
  if (MASK) {
    if (2 * t < lo || 2 * t >= rows) sv[0] = 0.f;
    if (2 * t + 1 < lo || 2 * t + 1 >= rows) sv[1] = 0.f;
    if (8 + 2 * t < lo || 8 + 2 * t >= rows) sv[2] = 0.f;
    if (9 + 2 * t < lo || 9 + 2 * t >= rows) sv[3] = 0.f;
  }
  const __half2 s01 = __floats2half2_rn(sv[0], sv[1]);
  const __half2 s23 = __floats2half2_rn(sv[2], sv[3]);
  const uint32_t sc01 = *reinterpret_cast<const uint32_t*>(&s01), sc23 = *reinterpret_cast<const uint32_t*>(&s23);

  // O += P . V~ over groups of 32 dims: this lane reads dims 32g + 4gr .. +3 of
  // tokens 2t, 2t+1, 8+2t, 9+2t and feeds n-tiles 4g .. 4g+3.
#pragma unroll
  for (int g = 0; g < C::VGROUPS; ++g) {
    const int ch = 2 * g + (gr >> 2);
    const uint32_t off = 4 * (gr & 3);
    const uint32_t wa = lds32(vt + i8_swz<D>(2 * t, ch) + off) ^ 0x80808080u;
    const uint32_t wb = lds32(vt + i8_swz<D>(2 * t + 1, ch) + off) ^ 0x80808080u;
    const uint32_t wc = lds32(vt + i8_swz<D>(2 * t + 8, ch) + off) ^ 0x80808080u;
    const uint32_t wd = lds32(vt + i8_swz<D>(2 * t + 9, ch) + off) ^ 0x80808080u;
    // Interleave the two tokens of each pair: [a_i, b_i, a_j, b_j].
    const uint32_t ab01 = __byte_perm(wa, wb, 0x5140), ab23 = __byte_perm(wa, wb, 0x7362);
    const uint32_t cd01 = __byte_perm(wc, wd, 0x5140), cd23 = __byte_perm(wc, wd, 0x7362);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t ab = i < 2 ? ab01 : ab23, cd = i < 2 ? cd01 : cd23;
      const uint32_t sel = (i & 1) ? 0x5342 : 0x5140;
      const uint32_t b0 = hmul2_u32(hsub2_u32(__byte_perm(ab, kF16Magic, sel), kF16Bias), sc01);
      const uint32_t b1 = hmul2_u32(hsub2_u32(__byte_perm(cd, kF16Magic, sel), kF16Bias), sc23);
      Mma<__half>::run(o[4 * g + i], a01, 0u, a23, 0u, b0, b1);
    }
  }
}

template <typename T, int D, int G, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32)
paged_decode_mma_int8_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap) {
  using C = I8Cfg<D, NW, STAGES>;
  static_assert(G >= 1 && G <= 8 && (G & (G - 1)) == 0, "groups of 1..8 query heads");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  wait_for_predecessor();
  const int g = blockIdx.x;
  const int s = long_first_seq<NW>(a, blockIdx.y), part = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq0 = g * a.group;
  const int gr = lane >> 2, t = lane & 3;

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
  if (L == 0) {
    T* o = static_cast<T*>(a.out) + (size_t(s) * a.num_q_heads + hq0) * D;
    for (int i = threadIdx.x; i < a.group * D / 8; i += NW * 32)
      reinterpret_cast<uint4*>(o)[i] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const int t0 = tr.aligned + part * a.part_tokens;
  const int ntok = min(L, t0 + a.part_tokens) - t0;
  const int nb = (ntok + kBlock - 1) / kBlock;
  const int head = part == 0 ? tr.first - tr.aligned : 0;

  unsigned char* ring = smem + size_t(warp) * STAGES * C::STAGE_BYTES;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t scale_s = smem_addr(smem + C::RING_BYTES) + warp * STAGES * C::SCALE_STAGE;
  const uint32_t bar_s = smem_addr(smem + C::RING_BYTES + C::SCALE_BYTES) + warp * STAGES * 8;
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < STAGES; ++st) mbar_init(bar_s + 8 * st, 1);
    mbar_init_fence();
  }
  __syncwarp();

  // Q~ of head hq0 + gr as the A operand, dims permuted per 16-dim chunk:
  // qa[c][0] = (dims 16c + 4t, +1), qa[c][1] = (dims 16c + 4t + 2, +3).
  uint32_t qa[C::KCHUNKS][2];
  float qmul;
  {
    float qf[C::KCHUNKS][4];
    float m = 0.f;
#pragma unroll
    for (int c = 0; c < C::KCHUNKS; ++c) {
      if (gr < a.group) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(
            static_cast<const T*>(a.q) + (size_t(s) * a.num_q_heads + hq0 + gr) * D + 16 * c + 4 * t));
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) qf[c][i] = float(e[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) qf[c][i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) m = fmaxf(m, fabsf(qf[c][i]));
    }
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
    // m < 2^E with E from m's exponent field (clamped for tiny or zero q);
    // scale by 2^(14 - E).
    const int E = max(int((__float_as_uint(m) >> 23) & 0xffu) - 126, -100);
    const float up = __uint_as_float(uint32_t(127 + 14 - E) << 23);
    qmul = a.scale_log2 * __uint_as_float(uint32_t(127 - 14 + E) << 23);
#pragma unroll
    for (int c = 0; c < C::KCHUNKS; ++c) {
      const __half2 h0 = __floats2half2_rn(qf[c][0] * up, qf[c][1] * up);
      const __half2 h1 = __floats2half2_rn(qf[c][2] * up, qf[c][3] * up);
      qa[c][0] = *reinterpret_cast<const uint32_t*>(&h0);
      qa[c][1] = *reinterpret_cast<const uint32_t*>(&h1);
    }
  }

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

  auto issue = [&](int k) {  // warp-uniform; k increases by one per call
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
      const uint32_t sdst = scale_s + st * C::SCALE_STAGE;
      const size_t row0 = (size_t(id) * a.num_kv_heads + g) * kBlock;
      mbar_arrive_expect_tx(bar, C::STAGE_BYTES + C::SCALE_STAGE);
#pragma unroll
      for (int j = 0; j < C::BOXES; ++j) {
        tma_load_2d(dst + j * C::BOX_BYTES, &kmap, C::BOX_COLS * j, int(row0), bar);
        tma_load_2d(dst + C::TILE_BYTES + j * C::BOX_BYTES, &vmap, C::BOX_COLS * j, int(row0), bar);
      }
      bulk_g2s(sdst, a.k_scale + row0, kBlock * 4, bar);
      bulk_g2s(sdst + kBlock * 4, a.v_scale + row0, kBlock * 4, bar);
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
    const uint32_t parity = (k / STAGES) & 1;
    const bool ok = mbar_wait_bounded(bar_s + 8 * st, parity);
    if (!__all_sync(kFull, ok)) {
      if (lane == 0) flag(a.status, PKV_DEV_WAIT_TIMEOUT);
      const int last = min(n_my, k + STAGES);
      for (int kk = k; kk < last; ++kk) mbar_wait_bounded(bar_s + 8 * (kk % STAGES), (kk / STAGES) & 1);
      break;
    }
    const int j = warp + k * NW;
    const int rows = min(kBlock, ntok - j * kBlock);
    const int lo = j == 0 ? head : 0;
    const uint32_t kt = ring_s + st * C::STAGE_BYTES;
    const uint32_t sc = scale_s + st * C::SCALE_STAGE;
    if (rows == kBlock && lo == 0)
      mma_tile_int8<D, NW, STAGES, false>(kt, kt + C::TILE_BYTES, sc, 0, rows, qa, o, mrun, lrun, qmul, lane);
    else
      mma_tile_int8<D, NW, STAGES, true>(kt, kt + C::TILE_BYTES, sc, lo, rows, qa, o, mrun, lrun, qmul, lane);
    __syncwarp();
    if (k + STAGES < n_my) issue(k + STAGES);
  }

  lrun += __shfl_xor_sync(kFull, lrun, 1);
  lrun += __shfl_xor_sync(kFull, lrun, 2);

  // Publish (acc[G][D], m[G], l[G]); n-tile 4q + i, column slot c holds dim 32q + 4c + i.
  float* wsm = reinterpret_cast<float*>(ring);
  if (gr < G) {
#pragma unroll
    for (int q = 0; q < C::VGROUPS; ++q) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        wsm[gr * D + 32 * q + 4 * (2 * t) + i] = o[4 * q + i][0];
        wsm[gr * D + 32 * q + 4 * (2 * t + 1) + i] = o[4 * q + i][1];
      }
    }
    if (t == 0) {
      wsm[G * D + gr] = mrun;
      wsm[G * D + G + gr] = lrun;
    }
  }
  __syncthreads();
  finish_chunk<T, D, G, NW>(a, smem, size_t(STAGES) * C::STAGE_BYTES, s, g, part, nparts);
}

}  // namespace pkv
