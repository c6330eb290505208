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
//    The contraction runs over a permuted order of the head dims: lane t
//    reads 16-byte chunks 2t, 2t+1 (and 2t+8, 2t+9 at D = 256; chunk t at
//    D = 64) of its two token rows with one 16-byte load each, and word r of
//    the q-th such chunk feeds k-slots 2t, 2t+1, 2t+8, 2t+9 of k-step 4q + r.
//  * O += P~ . C_V with P~ = p * s_V * 2^e rounded to fp16 once and the V
//    codes exact in fp16: the V scale of each token rides on its softmax
//    weight. e is a per-warp power of two that keeps every P~ below 2^14
//    (s_V below 2^(14 - e)): it only falls, when a tile brings a larger
//    scale, and the accumulator is rescaled by the same exact power of two
//    together with the softmax rescale. Each lane loads one 16-byte chunk
//    (8 bytes at D = 64) from each of its 4 token rows; column slot c of
//    n-tile j holds head dim 16c + j (8c + j at D = 64; n-tiles 16..31 at
//    D = 256: 128 + 16c + j - 16), which the epilogue undoes.
//  * K and V tiles arrive by TMA tensor copies of uint8 boxes (16 rows x
//    min(D, 128) bytes) with the 128-byte swizzle (64-byte at D = 64), which
//    keeps the 16-byte loads above free of bank conflicts (2-way for the V
//    loads at D = 64); the 16 K and 16 V scales of the tile arrive by two
//    64-byte bulk copies.
// Rounding P~ to fp16 adds at most 2^-11 relative error per term, far below
// the quantisation step of the codes.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "decode_mma.cuh"
#include "decode_prefix.cuh"

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

// 16-byte chunk of a code row that lane t reads for its q-th QK load, and the
// head dim that k-step c = 4q + r, word r, byte i of lane t stands for.
template <int D>
__device__ __forceinline__ int i8_k_chunk(int q, int t) {
  return D == 64 ? t : 2 * t + (q & 1) + 8 * (q >> 1);
}
// Head dim of column slot c of PV n-tile j (the permutation the V loads make).
template <int D>
__host__ __device__ constexpr int i8_v_dim(int j, int c) {
  return D == 64 ? 8 * c + j : 128 * (j / 16) + 16 * c + (j % 16);
}

// Running V-scale state of a warp: P~ = p * s_V * vmul with vmul = 2^(14 - E)
// for every s_V seen below vbound = 2^E.
struct VScale {
  float vbound = 0x1p-100f;
  float vmul = 0x1p114f;
};

template <int D, int NW, int STAGES, bool MASK>
__device__ __forceinline__ void mma_tile_int8(uint32_t kt, uint32_t vt, uint32_t st_scale, int lo, int rows,
                                              const uint32_t (&qa)[D / 16][2], float (&o)[D / 8][4],
                                              float& mrun, float& lrun, VScale& vs, float qmul, int lane,
                                              bool row_on = true) {
  using C = I8Cfg<D, NW, STAGES>;
  const int t = lane & 3, gr = lane >> 2;

  // S = Q~ . C_K^T: n-tile 0 = tokens 0..7 (this lane's token gr), n-tile 1 = tokens 8..15.
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int q = 0; q < C::KCHUNKS / 4; ++q) {
    const int ch = i8_k_chunk<D>(q, t);
    const uint4 w0 = lds128(kt + i8_swz<D>(gr, ch));
    const uint4 w1 = lds128(kt + i8_swz<D>(gr + 8, ch));
    const uint32_t a0[4] = {w0.x, w0.y, w0.z, w0.w}, a1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      uint32_t b0, b1, b2, b3;
      codes_to_f16x2(a0[r], b0, b1);
      codes_to_f16x2(a1[r], b2, b3);
      Mma<__half>::run(s0, qa[4 * q + r][0], 0u, qa[4 * q + r][1], 0u, b0, b1);
      Mma<__half>::run(s1, qa[4 * q + r][0], 0u, qa[4 * q + r][1], 0u, b2, b3);
    }
  }

  // Scores of head gr for tokens 2t, 2t+1, 8+2t, 9+2t, in the log2 domain.
  const float2 ka = lds_f32x2(st_scale + 8 * t);
  const float2 kb = lds_f32x2(st_scale + 32 + 8 * t);
  float x[4] = {s0[0] * ka.x * qmul, s0[1] * ka.y * qmul, s1[0] * kb.x * qmul, s1[1] * kb.y * qmul};
  // V scales of the same tokens; rows outside [lo, rows) get 0 (their stale
  // codes and scales then contribute exactly nothing).
  const float2 va = lds_f32x2(st_scale + 64 + 8 * t);
  const float2 vb = lds_f32x2(st_scale + 96 + 8 * t);
  float sv[4] = {va.x, va.y, vb.x, vb.y};
  if (MASK) {
    if (2 * t < lo || 2 * t >= rows) x[0] = -INFINITY, sv[0] = 0.f;
    if (2 * t + 1 < lo || 2 * t + 1 >= rows) x[1] = -INFINITY, sv[1] = 0.f;
    if (8 + 2 * t < lo || 8 + 2 * t >= rows) x[2] = -INFINITY, sv[2] = 0.f;
    if (9 + 2 * t < lo || 9 + 2 * t >= rows) x[3] = -INFINITY, sv[3] = 0.f;
  }
  if (!row_on) x[0] = x[1] = x[2] = x[3] = -INFINITY;  // this lane's row does not attend to this tile
  float mt = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
  mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
  const float mn = fmaxf(mrun, mt);
  const float mref = mn == -INFINITY ? 0.f : mn;  // a row with no valid score yet: weights exactly 0
  // The tile's largest V scale (the 16 tokens are spread over t), warp-uniform.
  float ms = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
  ms = fmaxf(ms, __shfl_xor_sync(kFull, ms, 1));
  ms = fmaxf(ms, __shfl_xor_sync(kFull, ms, 2));
  float vratio = 1.f;
  const bool vgrow = ms >= vs.vbound;
  if (vgrow) {  // ms in [2^(E-1), 2^E): vbound = 2^E, vmul = 2^(14 - E)
    const int E = min(max(int((__float_as_uint(ms) >> 23) & 0xffu) - 126, -99), 113);
    const float nmul = __uint_as_float(uint32_t(127 + 14 - E) << 23);
    vratio = nmul / vs.vmul;  // a power of two: exact
    vs.vmul = nmul;
    vs.vbound = __uint_as_float(uint32_t(127 + E) << 23);
  }
  if (vgrow || __any_sync(kFull, mn > mrun)) {
    const float alpha = fast_exp2(mrun - mref);  // 1 for rows whose max did not move
    lrun *= alpha;
    const float oa = alpha * vratio;
#pragma unroll
    for (int nd = 0; nd < C::NTILES; ++nd) {
      o[nd][0] *= oa;
      o[nd][1] *= oa;
    }
    mrun = mn;
  }
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = fast_exp2(x[i] - mref);
  lrun += (p[0] + p[1]) + (p[2] + p[3]);
  const __half2 p01 = __floats2half2_rn(p[0] * (sv[0] * vs.vmul), p[1] * (sv[1] * vs.vmul));
  const __half2 p23 = __floats2half2_rn(p[2] * (sv[2] * vs.vmul), p[3] * (sv[3] * vs.vmul));
  const uint32_t a01 = *reinterpret_cast<const uint32_t*>(&p01);
  const uint32_t a23 = *reinterpret_cast<const uint32_t*>(&p23);

  // O += P~ . C_V: this lane reads its 16-byte chunk (8 bytes at D = 64) of
  // tokens 2t, 2t+1, 8+2t, 9+2t and feeds column gr of every n-tile.
  constexpr int VW = D == 64 ? 8 : 16;        // bytes a lane takes from a row per load
  constexpr int VLOADS = D == 256 ? 2 : 1;    // loads per row
#pragma unroll
  for (int v = 0; v < VLOADS; ++v) {
    uint32_t wa[VW / 4], wb[VW / 4], wc[VW / 4], wd[VW / 4];
    if constexpr (D == 64) {
      const uint32_t off = 8 * (gr & 1);
      const uint2 xa = lds64(vt + i8_swz<D>(2 * t, gr >> 1) + off);
      const uint2 xb = lds64(vt + i8_swz<D>(2 * t + 1, gr >> 1) + off);
      const uint2 xc = lds64(vt + i8_swz<D>(2 * t + 8, gr >> 1) + off);
      const uint2 xd = lds64(vt + i8_swz<D>(2 * t + 9, gr >> 1) + off);
      wa[0] = xa.x, wa[1] = xa.y, wb[0] = xb.x, wb[1] = xb.y;
      wc[0] = xc.x, wc[1] = xc.y, wd[0] = xd.x, wd[1] = xd.y;
    } else {
      const int ch = 8 * v + gr;
      const uint4 xa = lds128(vt + i8_swz<D>(2 * t, ch));
      const uint4 xb = lds128(vt + i8_swz<D>(2 * t + 1, ch));
      const uint4 xc = lds128(vt + i8_swz<D>(2 * t + 8, ch));
      const uint4 xd = lds128(vt + i8_swz<D>(2 * t + 9, ch));
      wa[0] = xa.x, wa[1] = xa.y, wa[2] = xa.z, wa[3] = xa.w;
      wb[0] = xb.x, wb[1] = xb.y, wb[2] = xb.z, wb[3] = xb.w;
      wc[0] = xc.x, wc[1] = xc.y, wc[2] = xc.z, wc[3] = xc.w;
      wd[0] = xd.x, wd[1] = xd.y, wd[2] = xd.z, wd[3] = xd.w;
    }
#pragma unroll
    for (int w = 0; w < VW / 4; ++w) {
      // Interleave the two tokens of each pair: [a_i, b_i, a_j, b_j].
      const uint32_t xa = wa[w] ^ 0x80808080u, xb = wb[w] ^ 0x80808080u;
      const uint32_t xc = wc[w] ^ 0x80808080u, xd = wd[w] ^ 0x80808080u;
      const uint32_t ab01 = __byte_perm(xa, xb, 0x5140), ab23 = __byte_perm(xa, xb, 0x7362);
      const uint32_t cd01 = __byte_perm(xc, xd, 0x5140), cd23 = __byte_perm(xc, xd, 0x7362);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t ab = i < 2 ? ab01 : ab23, cd = i < 2 ? cd01 : cd23;
        const uint32_t sel = (i & 1) ? 0x5342 : 0x5140;
        const uint32_t b0 = hsub2_u32(__byte_perm(ab, kF16Magic, sel), kF16Bias);
        const uint32_t b1 = hsub2_u32(__byte_perm(cd, kF16Magic, sel), kF16Bias);
        Mma<__half>::run(o[VW * v + 4 * w + i], a01, 0u, a23, 0u, b0, b1);
      }
    }
  }
}

// Q~ of one query row as the A operand, dims permuted as the K loads are:
// k-step c = 4q + r takes dims d, d+1 (qa[c][0]) and d+2, d+3 (qa[c][1]),
// d = 16 * i8_k_chunk(q, t) + 4r; the row is scaled by a power of two that
// brings max|q| to [2^13, 2^14) (exact for bf16 and fp16 queries), and
// `qmul` = scale * log2(e) / that power. `qrow` null: a zero row.
template <typename T, int D>
__device__ __forceinline__ void i8_query(const T* qrow, int t, uint32_t (&qa)[D / 16][2], float& qmul,
                                         float scale_log2) {
  constexpr int KCHUNKS = D / 16;
  float qf[KCHUNKS][4];
  float m = 0.f;
#pragma unroll
  for (int c = 0; c < KCHUNKS; ++c) {
    if (qrow) {
      const int d0 = 16 * i8_k_chunk<D>(c / 4, t) + 4 * (c % 4);
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(qrow + d0));
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
  qmul = scale_log2 * __uint_as_float(uint32_t(127 - 14 + E) << 23);
#pragma unroll
  for (int c = 0; c < KCHUNKS; ++c) {
    const __half2 h0 = __floats2half2_rn(qf[c][0] * up, qf[c][1] * up);
    const __half2 h1 = __floats2half2_rn(qf[c][2] * up, qf[c][3] * up);
    qa[c][0] = *reinterpret_cast<const uint32_t*>(&h0);
    qa[c][1] = *reinterpret_cast<const uint32_t*>(&h1);
  }
}

// Publishes a warp's (acc[G][D], m[G], l[G]) at the start of its ring in
// head-dim order, with the V-scale power of two taken out (exact).
template <int D, int G>
__device__ __forceinline__ void i8_publish(float* wsm, const float (&o)[D / 8][4], float mrun, float lrun,
                                           const VScale& vs, int lane) {
  const int t = lane & 3, gr = lane >> 2;
  if (gr < G) {
    const float unmul = 1.f / vs.vmul;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      wsm[gr * D + i8_v_dim<D>(j, 2 * t)] = o[j][0] * unmul;
      wsm[gr * D + i8_v_dim<D>(j, 2 * t + 1)] = o[j][1] * unmul;
    }
    if (t == 0) {
      wsm[G * D + gr] = mrun;
      wsm[G * D + G + gr] = lrun;
    }
  }
}

// One query row per KV head (group size 1, head_dim <= 128): QK^T on the
// integer units instead of the tensor cores. The query becomes two int8
// digit planes, q ~ s1 * d1 + s2 * d2 with s1 = max|q| / 127, d1 = rint(q /
// s1), s2 = s1 / 254 and d2 = rint((q - s1 d1) / s2), so |q - (s1 d1 + s2
// d2)| <= max|q| / 64516, and each K code word meets each plane in one
// dp4a (four int8 products summed exactly in int32): no code is converted.
// Lane l takes token l / 2 and head dims [D/2 * (l & 1), D/2 * (l & 1 + 1)).
// PV stays on the tensor cores (the weights gathered into row 0 of the A
// operand), exactly as in mma_tile_int8.
template <int D>
struct MhaQuery {
  int p1[D / 8], p2[D / 8];  // this lane's half of the two planes, 4 dims a word
  float s1, s2;              // plane scales times scale * log2(e)
};

template <typename T, int D>
__device__ __forceinline__ void i8_query_mha(const T* qrow, int lane, float scale_log2, MhaQuery<D>& mq) {
  // Lane l digitises dims 4l .. 4l+3 (lanes past D/4 repeat the first ones),
  // then each lane gathers the words of its half by shuffles.
  constexpr int W = D / 8;  // words of one half
  const int wl = lane % (D / 4);
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(qrow + 4 * wl));
  const T* e = reinterpret_cast<const T*>(&u);
  float qf[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) qf[i] = float(e[i]);
  float m = fmaxf(fmaxf(fabsf(qf[0]), fabsf(qf[1])), fmaxf(fabsf(qf[2]), fabsf(qf[3])));
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  const float s1 = m / 127.f, s2 = s1 / 254.f;
  const float inv1 = m > 0.f ? 127.f / m : 0.f, inv2 = m > 0.f ? 254.f * 127.f / m : 0.f;
  uint32_t w1 = 0, w2 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float d1 = rintf(qf[i] * inv1);
    const float d2 = fminf(fmaxf(rintf((qf[i] - d1 * s1) * inv2), -127.f), 127.f);
    w1 |= (uint32_t(int(d1)) & 0xffu) << (8 * i);
    w2 |= (uint32_t(int(d2)) & 0xffu) << (8 * i);
  }
  const int h = lane & 1;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    mq.p1[w] = int(__shfl_sync(kFull, w1, W * h + w));
    mq.p2[w] = int(__shfl_sync(kFull, w2, W * h + w));
  }
  mq.s1 = s1 * scale_log2;
  mq.s2 = s2 * scale_log2;
}

template <int D, int NW, int STAGES, bool MASK>
__device__ __forceinline__ void mma_tile_int8_mha(uint32_t kt, uint32_t vt, uint32_t st_scale, int lo, int rows,
                                                  const MhaQuery<D>& mq, float (&o)[D / 16][4], float& mrun,
                                                  float& lsum, VScale& vs, int lane) {
  using C = I8Cfg<D, NW, STAGES>;
  static_assert(D <= 128, "the integer QK^T keeps a half row of both planes in registers");
  const int tk = lane >> 1, h = lane & 1;
  const int t = lane & 3, gr = lane >> 2;

  // S = q . C_K^T for token tk: this lane's half of the dims, then the pair's sum.
  int acc1 = 0, acc2 = 0;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    const uint4 w = lds128(kt + i8_swz<D>(tk, (D / 32) * h + c));
    acc1 = __dp4a(int(w.x), mq.p1[4 * c], acc1);
    acc2 = __dp4a(int(w.x), mq.p2[4 * c], acc2);
    acc1 = __dp4a(int(w.y), mq.p1[4 * c + 1], acc1);
    acc2 = __dp4a(int(w.y), mq.p2[4 * c + 1], acc2);
    acc1 = __dp4a(int(w.z), mq.p1[4 * c + 2], acc1);
    acc2 = __dp4a(int(w.z), mq.p2[4 * c + 2], acc2);
    acc1 = __dp4a(int(w.w), mq.p1[4 * c + 3], acc1);
    acc2 = __dp4a(int(w.w), mq.p2[4 * c + 3], acc2);
  }
  float sc = fmaf(mq.s1, float(acc1), mq.s2 * float(acc2));
  sc += __shfl_xor_sync(kFull, sc, 1);
  float x, sv;
  {
    float ks, vsc;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(ks) : "r"(st_scale + 4 * tk));
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(vsc) : "r"(st_scale + 64 + 4 * tk));
    x = sc * ks;
    sv = vsc;
  }
  if (MASK && (tk < lo || tk >= rows)) x = -INFINITY, sv = 0.f;
  // the tile's max score and largest V scale, over the 16 tokens (lanes 2 apart)
  float mt = x, ms = sv;
#pragma unroll
  for (int off = 2; off < 32; off <<= 1) {
    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, off));
    ms = fmaxf(ms, __shfl_xor_sync(kFull, ms, off));
  }
  const float mn = fmaxf(mrun, mt);
  const float mref = mn == -INFINITY ? 0.f : mn;
  float vratio = 1.f;
  const bool vgrow = ms >= vs.vbound;
  if (vgrow) {  // ms in [2^(E-1), 2^E): vbound = 2^E, vmul = 2^(14 - E)
    const int E = min(max(int((__float_as_uint(ms) >> 23) & 0xffu) - 126, -99), 113);
    const float nmul = __uint_as_float(uint32_t(127 + 14 - E) << 23);
    vratio = nmul / vs.vmul;
    vs.vmul = nmul;
    vs.vbound = __uint_as_float(uint32_t(127 + E) << 23);
  }
  if (vgrow || mn > mrun) {  // warp-uniform
    const float alpha = fast_exp2(mrun - mref);
    lsum *= alpha;
    const float oa = alpha * vratio;
#pragma unroll
    for (int nb = 0; nb < D / 16; ++nb) {  // column 0 of each block (columns 1..7 stay zero)
      o[nb][0] *= oa;
      o[nb][2] *= oa;
    }
    mrun = mn;
  }
  const float p = fast_exp2(x - mref);
  if (h == 0) lsum += p;  // each token once
  const float pv = p * (sv * vs.vmul);
  // Column 0 of the B operand: lanes 0..3 (gr = 0) take the weights of tokens 2t, 2t+1, 2t+8, 2t+9.
  const float w0 = __shfl_sync(kFull, pv, 4 * t), w1 = __shfl_sync(kFull, pv, 4 * t + 2);
  const float w2 = __shfl_sync(kFull, pv, 4 * t + 16), w3 = __shfl_sync(kFull, pv, 4 * t + 18);
  const __half2 p01 = __floats2half2_rn(w0, w1);
  const __half2 p23 = __floats2half2_rn(w2, w3);
  const uint32_t b01 = gr == 0 ? *reinterpret_cast<const uint32_t*>(&p01) : 0u;
  const uint32_t b23 = gr == 0 ? *reinterpret_cast<const uint32_t*>(&p23) : 0u;

  // O^T += C_V^T . P~ on the tensor cores: M = 16 head dims, K = the 16
  // tokens, N = 8 columns of which column 0 is the weights (lanes gr = 0 give
  // the B operand). This lane reads its 16-byte chunk (8 bytes at D = 64) of
  // tokens 2t, 2t+1, 8+2t, 9+2t; rows gr and gr + 8 of block b are head dims
  // VW * gr + 2b and VW * gr + 2b + 1.
  constexpr int VW = D == 64 ? 8 : 16;
  uint32_t wa[VW / 4], wb[VW / 4], wc[VW / 4], wd[VW / 4];
  if constexpr (D == 64) {
    const uint32_t off = 8 * (gr & 1);
    const uint2 xa = lds64(vt + i8_swz<D>(2 * t, gr >> 1) + off);
    const uint2 xb = lds64(vt + i8_swz<D>(2 * t + 1, gr >> 1) + off);
    const uint2 xc = lds64(vt + i8_swz<D>(2 * t + 8, gr >> 1) + off);
    const uint2 xd = lds64(vt + i8_swz<D>(2 * t + 9, gr >> 1) + off);
    wa[0] = xa.x, wa[1] = xa.y, wb[0] = xb.x, wb[1] = xb.y;
    wc[0] = xc.x, wc[1] = xc.y, wd[0] = xd.x, wd[1] = xd.y;
  } else {
    const uint4 xa = lds128(vt + i8_swz<D>(2 * t, gr));
    const uint4 xb = lds128(vt + i8_swz<D>(2 * t + 1, gr));
    const uint4 xc = lds128(vt + i8_swz<D>(2 * t + 8, gr));
    const uint4 xd = lds128(vt + i8_swz<D>(2 * t + 9, gr));
    wa[0] = xa.x, wa[1] = xa.y, wa[2] = xa.z, wa[3] = xa.w;
    wb[0] = xb.x, wb[1] = xb.y, wb[2] = xb.z, wb[3] = xb.w;
    wc[0] = xc.x, wc[1] = xc.y, wc[2] = xc.z, wc[3] = xc.w;
    wd[0] = xd.x, wd[1] = xd.y, wd[2] = xd.z, wd[3] = xd.w;
  }
#pragma unroll
  for (int w = 0; w < VW / 4; ++w) {
    // Interleave the two tokens of each pair: [a_i, b_i, a_j, b_j].
    const uint32_t xa = wa[w] ^ 0x80808080u, xb = wb[w] ^ 0x80808080u;
    const uint32_t xc = wc[w] ^ 0x80808080u, xd = wd[w] ^ 0x80808080u;
    const uint32_t ab01 = __byte_perm(xa, xb, 0x5140), ab23 = __byte_perm(xa, xb, 0x7362);
    const uint32_t cd01 = __byte_perm(xc, xd, 0x5140), cd23 = __byte_perm(xc, xd, 0x7362);
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // block 2w + half: bytes 2 half (row gr) and 2 half + 1 (row gr + 8)
      const uint32_t ab = half ? ab23 : ab01, cd = half ? cd23 : cd01;
      const uint32_t a0 = hsub2_u32(__byte_perm(ab, kF16Magic, 0x5140), kF16Bias);
      const uint32_t a1 = hsub2_u32(__byte_perm(ab, kF16Magic, 0x5342), kF16Bias);
      const uint32_t a2 = hsub2_u32(__byte_perm(cd, kF16Magic, 0x5140), kF16Bias);
      const uint32_t a3 = hsub2_u32(__byte_perm(cd, kF16Magic, 0x5342), kF16Bias);
      Mma<__half>::run(o[2 * w + half], a0, a1, a2, a3, b01, b23);
    }
  }
}

// Publishes a warp's (acc[1][D], m, l) of the one-query tile in head-dim
// order, with the V-scale power of two taken out (exact): column 0 of block
// b sits in lanes t = 0, rows gr and gr + 8 = head dims VW * gr + 2b, + 1.
template <int D>
__device__ __forceinline__ void i8_publish_mha(float* wsm, const float (&o)[D / 16][4], float mrun, float lrun,
                                               const VScale& vs, int lane) {
  constexpr int VW = D == 64 ? 8 : 16;
  const int t = lane & 3, gr = lane >> 2;
  if (t == 0) {
    const float unmul = 1.f / vs.vmul;
#pragma unroll
    for (int b = 0; b < D / 16; ++b) {
      wsm[VW * gr + 2 * b] = o[b][0] * unmul;
      wsm[VW * gr + 2 * b + 1] = o[b][2] * unmul;
    }
  }
  if (lane == 0) {
    wsm[D] = mrun;      // G = 1: m at acc[1][D], l after it
    wsm[D + 1] = lrun;
  }
}

// One CTA of the shared-prefix schedule over the INT8 cache (the 16-bit
// version, prefix_cta in decode_prefix.cuh, describes the chunk): the
// members' query rows share each K/V code tile, copied once.
template <typename T, int D, int G, int NW, int STAGES>
__device__ __forceinline__ void prefix_cta_int8(const DecodeArgs& a, const CUtensorMap& kmap,
                                                const CUtensorMap& vmap, unsigned char* smem, int ci) {
  using C = I8Cfg<D, NW, STAGES>;
  static_assert(G == kPrefixRows, "a group's rows fill the tile's G rows");
  const int g = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;
  PrefixChunk<NW> c;
  if (!c.init(a, ci, warp)) return;

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

  // Row r: query head g * group + r % group of member r / group.
  const int my_member = gr / a.group;
  uint32_t qa[C::KCHUNKS][2];
  float qmul;
  i8_query<T, D>(gr < c.rows ? static_cast<const T*>(a.q) +
                                   (size_t(c.s0 + my_member) * a.num_q_heads + g * a.group + gr % a.group) * D
                             : nullptr,
                 t, qa, qmul, a.scale_log2);

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
      const int st = k % STAGES;
      const uint32_t bar = bar_s + 8 * st;
      const uint32_t dst = ring_s + st * C::STAGE_BYTES;
      const uint32_t sdst = scale_s + st * C::SCALE_STAGE;
      const size_t row0 = (size_t(id) * a.num_kv_heads + g) * kBlock;
      mbar_arrive_expect_tx(bar, C::STAGE_BYTES + C::SCALE_STAGE);
#pragma unroll
      for (int jb = 0; jb < C::BOXES; ++jb) {
        tma_load_2d(dst + jb * C::BOX_BYTES, &kmap, C::BOX_COLS * jb, int(row0), bar);
        tma_load_2d(dst + C::TILE_BYTES + jb * C::BOX_BYTES, &vmap, C::BOX_COLS * jb, int(row0), bar);
      }
      bulk_g2s(sdst, a.k_scale + row0, kBlock * 4, bar);
      bulk_g2s(sdst + kBlock * 4, a.v_scale + row0, kBlock * 4, bar);
    }
  };

  float o[C::NTILES][4];
#pragma unroll
  for (int nd = 0; nd < C::NTILES; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float mrun = -INFINITY, lrun = 0.f;
  VScale vs;
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
    const uint32_t sc = scale_s + st * C::SCALE_STAGE;
    if (valid == kBlock)
      mma_tile_int8<D, NW, STAGES, false>(kt, kt + C::TILE_BYTES, sc, 0, kBlock, qa, o, mrun, lrun, vs, qmul,
                                          lane, row_on);
    else
      mma_tile_int8<D, NW, STAGES, true>(kt, kt + C::TILE_BYTES, sc, 0, valid, qa, o, mrun, lrun, vs, qmul, lane,
                                         row_on);
    __syncwarp();
    if (k + STAGES < n_my) issue(k + STAGES);
  }
  lrun += __shfl_xor_sync(kFull, lrun, 1);
  lrun += __shfl_xor_sync(kFull, lrun, 2);
  i8_publish<D, G>(reinterpret_cast<float*>(ring), o, mrun, lrun, vs, lane);
  __syncthreads();
  prefix_finish<T, D, G, NW>(a, c, smem, size_t(STAGES) * C::STAGE_BYTES);
}

template <typename T, int D, int G, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32, (G == 1 && D <= 128) ? 16 / NW : 0)  // one-query tile: 128 registers
paged_decode_mma_int8_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap) {
  using C = I8Cfg<D, NW, STAGES>;
  static_assert(G >= 1 && G <= 8 && (G & (G - 1)) == 0, "groups of 1..8 query heads");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  wait_for_predecessor();
  const int g = blockIdx.x;
  // Shared-prefix schedule: the plan's chunks take the first grid rows, the
  // sequences outside any group the next ones (as in the 16-bit kernel).
  int s;
  if (a.prefix_header) {
    const int4 ph = __ldg(a.prefix_header);
    const bool planned = ph.x == kPlanMagicPrefix && ph.y == a.num_seqs;
    const int nchunks = planned ? min(max(ph.z, 0), a.prefix_slots) : 0;
    const int nothers = planned ? min(max(ph.w, 0), a.num_seqs) : a.num_seqs;
    if (!planned && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) flag(a.status, PKV_DEV_BAD_PLAN);
    if constexpr (G == kPrefixRows) {
      if (int(blockIdx.y) < nchunks) {
        prefix_cta_int8<T, D, G, NW, STAGES>(a, kmap, vmap, smem, int(blockIdx.y));
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
    s = long_first_seq<NW>(a, blockIdx.y);
  }
  const int part = blockIdx.z;
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

  // Group size 1 up to head_dim 128: QK^T on the integer units against the
  // query's two digit planes (mma_tile_int8_mha); otherwise Q~ of head hq0 + gr
  // as the tensor cores' A operand (rows past the group zero).
  constexpr bool kMha = G == 1 && D <= 128;
  uint32_t qa[C::KCHUNKS][2];
  float qmul = 0.f;
  MhaQuery<D <= 128 ? D : 128> mq;
  if constexpr (kMha) {
    i8_query_mha<T, D>(static_cast<const T*>(a.q) + (size_t(s) * a.num_q_heads + hq0) * D, lane, a.scale_log2, mq);
  } else {
    i8_query<T, D>(gr < a.group ? static_cast<const T*>(a.q) + (size_t(s) * a.num_q_heads + hq0 + gr) * D
                                : nullptr,
                   t, qa, qmul, a.scale_log2);
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

  constexpr int OROWS = kMha ? D / 16 : C::NTILES;  // accumulator blocks
  float o[OROWS][4];
#pragma unroll
  for (int nd = 0; nd < OROWS; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float mrun = -INFINITY, lrun = 0.f;
  VScale vs;

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
    if constexpr (kMha) {
      if (rows == kBlock && lo == 0)
        mma_tile_int8_mha<D, NW, STAGES, false>(kt, kt + C::TILE_BYTES, sc, 0, rows, mq, o, mrun, lrun, vs, lane);
      else
        mma_tile_int8_mha<D, NW, STAGES, true>(kt, kt + C::TILE_BYTES, sc, lo, rows, mq, o, mrun, lrun, vs, lane);
    } else {
      if (rows == kBlock && lo == 0)
        mma_tile_int8<D, NW, STAGES, false>(kt, kt + C::TILE_BYTES, sc, 0, rows, qa, o, mrun, lrun, vs, qmul, lane);
      else
        mma_tile_int8<D, NW, STAGES, true>(kt, kt + C::TILE_BYTES, sc, lo, rows, qa, o, mrun, lrun, vs, qmul, lane);
    }
    __syncwarp();
    if (k + STAGES < n_my) issue(k + STAGES);
  }

  if constexpr (kMha) {  // each lane summed the weights of its own token's tiles (h == 0 lanes only)
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) lrun += __shfl_xor_sync(kFull, lrun, off);
  } else {
    lrun += __shfl_xor_sync(kFull, lrun, 1);
    lrun += __shfl_xor_sync(kFull, lrun, 2);
  }

  if constexpr (kMha)
    i8_publish_mha<D>(reinterpret_cast<float*>(ring), o, mrun, lrun, vs, lane);
  else
    i8_publish<D, G>(reinterpret_cast<float*>(ring), o, mrun, lrun, vs, lane);
  __syncthreads();
  finish_chunk<T, D, G, NW>(a, smem, size_t(STAGES) * C::STAGE_BYTES, s, g, part, nparts);
}

}  // namespace pkv
