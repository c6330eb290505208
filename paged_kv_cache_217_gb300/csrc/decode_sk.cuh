// PagedAttention decode with a balanced persistent schedule (sm_103a).
//
// Computes the same thing as decode.cuh (ordinary softmax attention of each
// sequence's query heads over its paged KV, per the abeam.tech summary of
// "Efficient Memory Management for Large Language Model Serving with
// PagedAttention", sections "技術の仕組み" and "よくある質問"), with a schedule
// that keeps every warp streaming until the whole batch is done:
//
//  * Work is the flattened sequence of 16-token tiles over (sequence s, KV head
//    g, tile j), s-major. Each CTA computes the prefix sums of the sequences'
//    tile counts in shared memory; warp w of the W persistent warps takes the
//    contiguous tile range [w*T/W, (w+1)*T/W). Every warp reads the same
//    number of KV bytes (to one tile), whatever the length mix.
//  * A warp walks its range through a private ring of shared-memory stages.
//    Tile copies (and, with a segment's first tile, the segment's q rows) are
//    issued STAGES ahead across (sequence, head) boundaries, so the ring never
//    drains between items; the block ids of the next 32 tiles are resolved
//    (binary search in the prefix sums, table read, bounds check) one batch
//    ahead by the 32 lanes in parallel.
//  * A range covers whole items and at most two partial ones (its first and
//    last). A whole item is normalised and written by its warp. A partial item
//    writes (max, sum, unnormalised V sum) to a workspace slot and bumps the
//    item's arrival counter (release/acquire at GPU scope); the last warp to
//    arrive merges the slots by log-sum-exp and writes the output.
//  * Tile math is unchanged: decode_tile (CUDA cores, G = 1) or mma_tile
//    (tensor cores, GQA groups).
#pragma once

#include "decode.cuh"
#include "decode_mma.cuh"

namespace pkv {

// Ring shape of the head_dim-128 configurations (the common case): warps per
// CTA (CUDA-core and tensor-core tiles) and stages per warp.
constexpr int kSkWarpsCuda = 6;
constexpr int kSkWarpsMma = 5;
constexpr int kSkStages = 2;

constexpr int kSkMaxSeqs = 2048;      // batch limit of the schedule (prefix sums in shared memory)
constexpr int kSkMaxWarps = 2048;     // partial slots: two per persistent warp
constexpr int kSkMinTilesPerWarp = 4; // small batches use fewer warps
constexpr size_t kSmemPerCta = 227 * 1024;

struct SkArgs {
  void* out;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* slots;            // [2 * kSkMaxWarps][slot_floats]: acc[group][D], m[group], l[group]
  unsigned int* counters;  // [S][Hkv] segments arrived; zero at launch
  unsigned int* status;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int max_blocks_per_seq;
  int num_blocks;
  int slot_floats;
  float scale_log2;
};

template <typename T, int D, int G, bool MMA>
struct SkCfg {
  static constexpr int ROW_BYTES = D * 2;
  // MMA tiles arrive as 128-byte-swizzled boxes (16 rows x 64 columns).
  static constexpr int TILE_BYTES = MMA ? (D / 64) * kBlock * 128 : kBlock * ROW_BYTES;
  static constexpr int Q_BYTES = G * D * 2;
  static constexpr int Q_SLOT = MMA ? ((Q_BYTES + 1023) / 1024) * 1024 : Q_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES + Q_SLOT;  // K tile, V tile, q rows
};

// Warps per CTA of the balanced schedule: rings of 2 stages per warp sized so
// that two CTAs (with their prefix sums and alignment slack) share an SM.
template <int D>
constexpr int sk_stages() {
  return D == 128 ? kSkStages : 2;
}
template <int D, int G>
constexpr int sk_warps() {
  constexpr int want = G == 1 ? (D == 256 ? 3 : (D == 128 ? kSkWarpsCuda : 6))
                              : (D == 64 ? 6 : (D == 128 ? kSkWarpsMma : 2));
  // at most what fits with room for 256 sequences of prefix sums
  constexpr int fit = int((kSmemPerCta - 1024 - 257 * sizeof(int)) /
                          (size_t(sk_stages<D>()) * (SkCfg<__half, D, G, (G > 1)>::STAGE_BYTES + 8)));
  return want < fit ? want : fit;
}

template <typename T, int D, int G, int NW, int STAGES, bool MMA>
struct SkSmem {
  using C = SkCfg<T, D, G, MMA>;
  static constexpr size_t RING = size_t(NW) * STAGES * C::STAGE_BYTES;
  static constexpr size_t BARS = size_t(NW) * STAGES * 8;
  static constexpr size_t bytes(int num_seqs) { return 1024 + RING + BARS + size_t(num_seqs + 1) * sizeof(int); }
  // Largest batch whose prefix sums still fit next to the rings.
  static constexpr int max_seqs() {
    const long long room = (long long)kSmemPerCta - 1024 - (long long)(RING + BARS) - (long long)sizeof(int);
    const long long n = room / (long long)sizeof(int);
    return n < kSkMaxSeqs ? int(n) : kSkMaxSeqs;
  }
  static_assert(1024 + RING + BARS + 256 * sizeof(int) <= kSmemPerCta, "rings must leave room for prefix sums");
};

__device__ __forceinline__ unsigned int atomic_add_acq_rel_gpu(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Packed per-tile metadata: s (16 bits), g (9 bits), rows-1 (4 bits),
// first-of-item (1 bit), last-of-item (1 bit).
struct TileMeta {
  int s, g, rows;
  bool item_first, item_last;
  static __device__ __forceinline__ uint32_t pack(int s, int g, int rows, bool f, bool l) {
    return uint32_t(s) | (uint32_t(g) << 16) | (uint32_t(rows - 1) << 25) | (uint32_t(f) << 29) |
           (uint32_t(l) << 30);
  }
  static __device__ __forceinline__ TileMeta unpack(uint32_t m) {
    TileMeta t;
    t.s = int(m & 0xffffu);
    t.g = int((m >> 16) & 0x1ffu);
    t.rows = int((m >> 25) & 0xfu) + 1;
    t.item_first = (m >> 29) & 1u;
    t.item_last = (m >> 30) & 1u;
    return t;
  }
};

// Merges the partial slots of item (s, g) -- written by warps wf..wl -- and
// writes the normalised output. Run by one warp.
template <typename T, int D>
__device__ __forceinline__ void sk_merge_item(const SkArgs& a, int s, int g, long long wf, long long wl,
                                              bool wf_head, int lane) {
  const int ng = a.group;
  T* out = static_cast<T*>(a.out) + (size_t(s) * a.num_q_heads + size_t(g) * ng) * D;
  for (int i = lane; i < ng * (D / 4); i += 32) {
    const int h = i / (D / 4), c4 = i % (D / 4);
    float M = -INFINITY;
    for (long long w = wf; w <= wl; ++w) {
      const long long slot = (w == wf && !wf_head) ? kSkMaxWarps + w : w;
      M = fmaxf(M, __ldcg(a.slots + slot * a.slot_floats + ng * D + h));
    }
    float den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long w = wf; w <= wl; ++w) {
      const long long slot = (w == wf && !wf_head) ? kSkMaxWarps + w : w;
      const float* sl = a.slots + slot * a.slot_floats;
      const float wt = fast_exp2(__ldcg(sl + ng * D + h) - M);
      den = fmaf(wt, __ldcg(sl + ng * D + ng + h), den);
      const float4 x = __ldcg(reinterpret_cast<const float4*>(sl + h * D) + c4);
      num.x = fmaf(wt, x.x, num.x);
      num.y = fmaf(wt, x.y, num.y);
      num.z = fmaf(wt, x.z, num.z);
      num.w = fmaf(wt, x.w, num.w);
    }
    const float inv = 1.f / den;
    T* o = out + h * D + c4 * 4;
    if constexpr (std::is_same<T, __half>::value) {
      reinterpret_cast<__half2*>(o)[0] = __floats2half2_rn(num.x * inv, num.y * inv);
      reinterpret_cast<__half2*>(o)[1] = __floats2half2_rn(num.z * inv, num.w * inv);
    } else {
      reinterpret_cast<__nv_bfloat162*>(o)[0] = __floats2bfloat162_rn(num.x * inv, num.y * inv);
      reinterpret_cast<__nv_bfloat162*>(o)[1] = __floats2bfloat162_rn(num.z * inv, num.w * inv);
    }
  }
}

template <typename T, int D, int G, int NW, int STAGES, bool MMA>
__global__ void __launch_bounds__(NW * 32)
paged_decode_sk_kernel(const SkArgs a, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap) {
  using C = SkCfg<T, D, G, MMA>;
  using SM = SkSmem<T, D, G, NW, STAGES, MMA>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* cum = reinterpret_cast<int*>(smem + SM::RING + SM::BARS);  // [S + 1] tiles before sequence s

  wait_for_predecessor();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.num_seqs, H = a.num_kv_heads;
  const int max_len = a.max_blocks_per_seq * kBlock;

  // ---- prefix sums of tile counts; zeros for empty sequences ------------------
  auto clamped_len = [&](int s) {
    const int L = __ldg(a.context_lens + s);
    return L < 0 ? 0 : (L > max_len ? max_len : L);
  };
  for (int s = threadIdx.x; s < S; s += NW * 32) {
    const int L = __ldg(a.context_lens + s);
    if ((L < 0 || L > max_len) && blockIdx.x == 0) flag(a.status, PKV_DEV_BAD_CONTEXT_LEN);
    cum[s + 1] = (clamped_len(s) + kBlock - 1) / kBlock;
  }
  __syncthreads();
  if (warp == 0) {  // inclusive scan of cum[1..S] by one warp, 32 values per step
    int carry = 0;
    for (int base = 0; base < S; base += 32) {
      const int i = base + lane;
      int v = i < S ? cum[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += n;
      }
      if (i < S) cum[i + 1] = v + carry;
      carry += __shfl_sync(kFull, v, 31);
    }
    if (lane == 0) cum[0] = 0;
  }
  __syncthreads();
  for (int s = blockIdx.x; s < S; s += gridDim.x) {  // L == 0: zero output rows
    if (cum[s + 1] == cum[s] && warp == 0) {
      T* o = static_cast<T*>(a.out) + size_t(s) * a.num_q_heads * D;
      for (int i = lane; i < a.num_q_heads * D / 8; i += 32) reinterpret_cast<uint4*>(o)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  const long long T_all = (long long)cum[S] * H;
  long long Wt = (long long)gridDim.x * NW;
  const long long w_cap = (T_all + kSkMinTilesPerWarp - 1) / kSkMinTilesPerWarp;
  if (Wt > w_cap) Wt = w_cap > 0 ? w_cap : 1;
  const long long gw = (long long)blockIdx.x * NW + warp;
  if (gw >= Wt || T_all == 0) return;
  const long long u0 = gw * T_all / Wt, u1 = (gw + 1) * T_all / Wt;
  const int n = int(u1 - u0);
  if (n <= 0) return;

  // ---- per-warp ring -----------------------------------------------------------
  unsigned char* ring = smem + size_t(warp) * STAGES * C::STAGE_BYTES;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar_s = smem_addr(smem + SM::RING) + warp * STAGES * 8;
  // q slots past the real group stay zero (the padded MMA rows / padded heads).
  if (a.group < G) {
    for (int st = 0; st < STAGES; ++st) {
      unsigned char* qs = ring + st * C::STAGE_BYTES + 2 * C::TILE_BYTES;
      for (int i = lane; i < (G - a.group) * D / 8; i += 32)
        reinterpret_cast<uint4*>(qs + a.group * D * 2)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < STAGES; ++st) mbar_init(bar_s + 8 * st, 1);
    mbar_init_fence();
  }
  __syncwarp();

  // ---- tile metadata, resolved 32 tiles at a time -------------------------------
  auto resolve = [&](int batch, int& id_out) -> uint32_t {
    const int k = batch * 32 + lane;
    id_out = 0;
    if (k >= n) return 0u;
    const long long u = u0 + k;
    int lo = 0, hi = S;  // largest s with cum[s] * H <= u
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if ((long long)cum[mid] * H <= u) lo = mid; else hi = mid;
    }
    const int s = lo;
    const int nbs = cum[s + 1] - cum[s];
    const long long off = u - (long long)cum[s] * H;
    const int g = int(off / nbs), j = int(off % nbs);
    int id = __ldg(a.block_tables + size_t(s) * a.max_blocks_per_seq + j);
    if (id < 0 || id >= a.num_blocks) {
      flag(a.status, PKV_DEV_BAD_BLOCK_ID);
      id = 0;
    }
    id_out = id;
    const int rows = min(kBlock, clamped_len(s) - j * kBlock);
    return TileMeta::pack(s, g, rows, j == 0, j == nbs - 1);
  };
  int id_cur, id_nxt;
  uint32_t meta_cur = resolve(0, id_cur);
  uint32_t meta_nxt = n > 32 ? resolve(1, id_nxt) : 0u;
  int cur_batch = 0;  // batch held in (meta_cur, id_cur); (meta_nxt, id_nxt) holds the next

  auto meta_of = [&](int k, int& id) -> uint32_t {  // k in the current or the next batch
    const bool nx = (k >> 5) != cur_batch;
    const uint32_t m = __shfl_sync(kFull, nx ? meta_nxt : meta_cur, k & 31);
    id = __shfl_sync(kFull, nx ? id_nxt : id_cur, k & 31);
    return m;
  };

  const char* kbase = static_cast<const char*>(a.k_pool);
  const char* vbase = static_cast<const char*>(a.v_pool);
  auto issue = [&](int k) {  // warp-uniform
    int id;
    const TileMeta tm = TileMeta::unpack(meta_of(k, id));
    if (lane == 0) {
      const int st = k % STAGES;
      const uint32_t bar = bar_s + 8 * st;
      const uint32_t dst = ring_s + st * C::STAGE_BYTES;
      const bool seg_first = tm.item_first || k == 0;
      const uint32_t qbytes = seg_first ? uint32_t(a.group) * D * 2 : 0u;
      if constexpr (MMA) {
        mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES + qbytes);
        const int y = (id * H + tm.g) * kBlock;
#pragma unroll
        for (int jb = 0; jb < D / 64; ++jb) {
          tma_load_2d(dst + jb * kBlock * 128, &kmap, 64 * jb, y, bar);
          tma_load_2d(dst + C::TILE_BYTES + jb * kBlock * 128, &vmap, 64 * jb, y, bar);
        }
      } else {
        const uint32_t bytes = uint32_t(tm.rows) * C::ROW_BYTES;
        mbar_arrive_expect_tx(bar, 2 * bytes + qbytes);
        const size_t off = (size_t(id) * H + tm.g) * C::TILE_BYTES;
        bulk_g2s(dst, kbase + off, bytes, bar);
        bulk_g2s(dst + C::TILE_BYTES, vbase + off, bytes, bar);
      }
      if (seg_first) {
        const T* qsrc = static_cast<const T*>(a.q) + (size_t(tm.s) * a.num_q_heads + size_t(tm.g) * a.group) * D;
        bulk_g2s(dst + 2 * C::TILE_BYTES, qsrc, qbytes, bar);
      }
    }
  };

  // ---- segment state -------------------------------------------------------------
  constexpr int LPR = D / 8;
  const int sub = lane & (LPR - 1), r = lane / LPR;  // CUDA-core lane split
  const int gr = lane >> 2, t4 = lane & 3;           // MMA fragment row / column pair
  float qf[MMA ? 1 : G][8];
  float acc[MMA ? 1 : G][8], lsum[MMA ? 1 : G], mrun[MMA ? 1 : G];
  uint32_t qa[MMA ? D / 16 : 1][2];
  float o[MMA ? D / 8 : 1][4];
  float mr1 = -INFINITY, lr1 = 0.f;
  bool seg_whole_start = false, seg_at_range_start = false;
  int seg_s = 0, seg_g = 0;

  const int pre = n < STAGES ? n : STAGES;
  for (int k = 0; k < pre; ++k) issue(k);

  for (int k = 0; k < n; ++k) {
    const int st = k % STAGES;
    const uint32_t parity = (k / STAGES) & 1;
    if ((k >> 5) != cur_batch) {  // move to the next batch, resolve the one after
      meta_cur = meta_nxt;
      id_cur = id_nxt;
      ++cur_batch;
      meta_nxt = (cur_batch + 1) * 32 < n ? resolve(cur_batch + 1, id_nxt) : 0u;
    }
    int id_unused;
    const TileMeta tm = TileMeta::unpack(meta_of(k, id_unused));
    const bool seg_first = tm.item_first || k == 0;
    const bool seg_last = tm.item_last || k == n - 1;

    const bool ok = mbar_wait_bounded(bar_s + 8 * st, parity);
    if (!__all_sync(kFull, ok)) {
      if (lane == 0) flag(a.status, PKV_DEV_WAIT_TIMEOUT);
      const int last = min(n, k + STAGES);
      for (int kk = k; kk < last; ++kk) mbar_wait_bounded(bar_s + 8 * (kk % STAGES), (kk / STAGES) & 1);
      return;
    }
    const uint32_t kt = ring_s + st * C::STAGE_BYTES;
    const uint32_t vt = kt + C::TILE_BYTES;
    const uint32_t qs = kt + 2 * C::TILE_BYTES;

    if (seg_first) {  // new segment: fresh state, q from this stage
      seg_whole_start = tm.item_first;
      seg_at_range_start = k == 0;
      seg_s = tm.s;
      seg_g = tm.g;
      if constexpr (MMA) {
        // Rows gr < G come from the q slot (zero past the real group); rows G..7
        // and 8..15 of the A operand are padding.
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          qa[ks][0] = qa[ks][1] = 0u;
          if (gr < G) {
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(qa[ks][0]) : "r"(qs + (gr * D + 16 * ks + 2 * t4) * 2));
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(qa[ks][1]) : "r"(qs + (gr * D + 16 * ks + 8 + 2 * t4) * 2));
          }
        }
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
        mr1 = -INFINITY;
        lr1 = 0.f;
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          Vec8<T>::to_float(lds128(qs + (h * D + sub * 8) * 2), qf[h]);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            qf[h][c] *= a.scale_log2;
            acc[h][c] = 0.f;
          }
          lsum[h] = 0.f;
          mrun[h] = -INFINITY;
        }
      }
    }

    if constexpr (MMA) {
      if (tm.rows == kBlock) {
        mma_tile<T, D, NW, STAGES, false>(kt, vt, 0, tm.rows, qa, o, mr1, lr1, a.scale_log2, lane);
      } else {
        zero_rows_outside<D>(vt, 0, tm.rows, lane);
        mma_tile<T, D, NW, STAGES, true>(kt, vt, 0, tm.rows, qa, o, mr1, lr1, a.scale_log2, lane);
      }
    } else {
      if (tm.rows == kBlock)
        decode_tile<T, D, G, NW, STAGES, false>(kt, vt, 0, tm.rows, qf, acc, lsum, mrun, lane);
      else
        decode_tile<T, D, G, NW, STAGES, true>(kt, vt, 0, tm.rows, qf, acc, lsum, mrun, lane);
    }
    __syncwarp();
    if (k + STAGES < n) issue(k + STAGES);

    if (!seg_last) continue;

    // ---- segment end: row sums across the lanes that share a row ---------------
    if constexpr (MMA) {
      lr1 += __shfl_xor_sync(kFull, lr1, 1);
      lr1 += __shfl_xor_sync(kFull, lr1, 2);
    } else {
#pragma unroll
      for (int m = LPR; m < 32; m <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          lsum[h] += __shfl_xor_sync(kFull, lsum[h], m);
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[h][c] += __shfl_xor_sync(kFull, acc[h][c], m);
        }
      }
    }
    const bool whole = seg_whole_start && tm.item_last;
    const size_t orow = size_t(seg_s) * a.num_q_heads + size_t(seg_g) * a.group;
    if (whole) {  // the item is entirely this warp's: normalise and write
      if constexpr (MMA) {
        if (gr < a.group) {
          const float inv = 1.f / lr1;
          T* orow_p = static_cast<T*>(a.out) + (orow + gr) * D;
#pragma unroll
          for (int nd = 0; nd < D / 8; ++nd) {
            float xr, yr;
            const uint32_t pk = Mma<T>::pack(o[nd][0] * inv, o[nd][1] * inv, xr, yr);
            *reinterpret_cast<uint32_t*>(orow_p + 8 * nd + 2 * t4) = pk;
          }
        }
      } else if (r == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (h < a.group) {
            const float inv = 1.f / lsum[h];
            float v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) v[c] = acc[h][c] * inv;
            reinterpret_cast<uint4*>(static_cast<T*>(a.out) + (orow + h) * D)[sub] = Vec8<T>::from_float(v);
          }
        }
      }
      continue;
    }

    // ---- partial item: slot, arrival counter, last arrival merges ---------------
    // A segment that starts at the range start uses this warp's head slot, any
    // other partial segment (it ends the range) its tail slot.
    const long long slot = seg_at_range_start ? gw : kSkMaxWarps + gw;
    float* sl = a.slots + slot * a.slot_floats;
    const int ng = a.group;
    if constexpr (MMA) {
      if (gr < ng) {
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd)
          *reinterpret_cast<float2*>(sl + gr * D + 8 * nd + 2 * t4) = make_float2(o[nd][0], o[nd][1]);
        if (t4 == 0) {
          sl[ng * D + gr] = mr1;
          sl[ng * D + ng + gr] = lr1;
        }
      }
    } else {
      if (r == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (h < ng) {
            float4* d4 = reinterpret_cast<float4*>(sl + h * D + sub * 8);
            d4[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
            d4[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
            if (sub == 0) {
              sl[ng * D + h] = mrun[h];
              sl[ng * D + ng + h] = lsum[h];
            }
          }
        }
      }
    }
    __syncwarp();
    // Warps covering the item: wf holds its first tile, wl its last.
    const int nbs = cum[seg_s + 1] - cum[seg_s];
    const long long u_first = (long long)cum[seg_s] * H + (long long)seg_g * nbs;
    const long long u_last = u_first + nbs - 1;
    const long long wf = ((u_first + 1) * Wt + T_all - 1) / T_all - 1;
    const long long wl = ((u_last + 1) * Wt + T_all - 1) / T_all - 1;
    unsigned int* counter = a.counters + size_t(seg_s) * H + seg_g;
    unsigned int arrived = 0;
    if (lane == 0) arrived = atomic_add_acq_rel_gpu(counter, 1u);
    arrived = __shfl_sync(kFull, arrived, 0);
    if (arrived == unsigned(wl - wf)) {  // last of the wl - wf + 1 segments
      __syncwarp();
      const bool wf_head = u_first == wf * T_all / Wt;
      sk_merge_item<T, D>(a, seg_s, seg_g, wf, wl, wf_head, lane);
      if (lane == 0) *counter = 0u;
    }
  }
}

}  // namespace pkv
