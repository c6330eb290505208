"""INT8 KV cache: per-row quantisation, the quantised cache write and decode over
the dequantised cache.

Test infrastructure (see the package docstring).

The glossary entry "PagedAttention（ページドアテンション）" (section
"他のKVキャッシュ最適化との組み合わせ") names INT8 KV-cache quantisation as a
companion of paging: it halves the size of a block at some cost in accuracy.
It gives no scheme. Reading taken (symmetric, one scale per stored row):

* Every (block, KV head, slot) row of K and of V gets its own fp32 scale
  s = max|x| / 127 and int8 codes c = rint(x / s) (ties to even), so that
  x ~= c * s with |x - c * s| <= s / 2. A row of zeros has s = 0 and codes 0.
  The codes are an integer decision taken in fp32 (IEEE division, as the
  kernel does), so both sides agree bit for bit.
* Decode over an INT8 cache is ordinary attention over the dequantised rows
  K = c_K * s_K and V = c_V * s_V (oracle.attention on those values).

Layouts: codes int8 [num_blocks, num_kv_heads, 16, head_dim]; scales fp32
[num_blocks, num_kv_heads, 16].
"""

import numpy as np

from .attention import attend, gather_kv
from .numerics import to_f64

BLOCK_SIZE = 16


def quantize_rows(x):
    """fp32 rows (last axis) -> (int8 codes, fp32 scales) as described above."""
    x = np.asarray(x, dtype=np.float32)
    m = np.max(np.abs(x), axis=-1)
    s = (m / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        c = np.rint(x / s[..., None])
    c = np.where(s[..., None] > 0, c, 0.0)
    c = np.clip(c, -127, 127).astype(np.int8)
    return c, s


def reshape_and_cache_int8(k, v, dtype, k_codes, v_codes, k_scale, v_scale, slot_mapping,
                           block_size=BLOCK_SIZE):
    """Quantise each new token's K/V rows and write codes and scales at its slot.

    k, v: [T, Hkv, D] fp16 (or bf16 bits); returns new (k_codes, v_codes,
    k_scale, v_scale) arrays. Negative slots are skipped.
    """
    kc, vc = np.array(k_codes, copy=True), np.array(v_codes, copy=True)
    ks, vs = np.array(k_scale, copy=True), np.array(v_scale, copy=True)
    kq, kqs = quantize_rows(to_f64(k, dtype).astype(np.float32))
    vq, vqs = quantize_rows(to_f64(v, dtype).astype(np.float32))
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        block, off = divmod(int(slot), block_size)
        kc[block, :, off] = kq[t]
        vc[block, :, off] = vq[t]
        ks[block, :, off] = kqs[t]
        vs[block, :, off] = vqs[t]
    return kc, vc, ks, vs


def dequantize(codes, scales):
    """float64 rows c * s."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def paged_attention_decode_int8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens,
                                scale, num_kv_heads, dtype, block_size=BLOCK_SIZE):
    """Decode attention over the dequantised INT8 cache, float64 [S, Hq, D]."""
    qf = to_f64(q, dtype)
    num_seqs, num_q_heads, head_dim = qf.shape
    group = num_q_heads // num_kv_heads
    kf = dequantize(k_codes, k_scale)
    vf = dequantize(v_codes, v_scale)
    out = np.zeros((num_seqs, num_q_heads, head_dim))
    for s in range(num_seqs):
        L = int(context_lens[s])
        for g in range(num_kv_heads):
            K = gather_kv(kf, block_tables[s], L, g, block_size)
            V = gather_kv(vf, block_tables[s], L, g, block_size)
            for h in range(g * group, (g + 1) * group):
                out[s, h] = attend(qf[s, h], K, V, scale)
    return out
