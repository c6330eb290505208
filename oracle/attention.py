"""Decode attention over a paged KV cache, as the plain definition, in float64.

Test infrastructure (see the package docstring).

What is computed. The pages are explicit that PagedAttention changes where
the K/V vectors live and how the kernel reaches them, not the attention
formula: the abeam.tech summary ("よくある質問": not a new formula) and the
pro-knowledge-base FAQ (accuracy unchanged). So the oracle gathers each
sequence's K and V through its block table into contiguous arrays and then
applies ordinary single-query softmax attention:

    out[s, h] = softmax(scale * K_s @ q[s, h]) @ V_s

Layout (shared with the CUDA path only as a documented contract, no code):
    q, out        : [num_seqs, num_q_heads, head_dim]
    k_pool, v_pool: [num_blocks, num_kv_heads, block_size, head_dim]
    block_tables  : int32 [num_seqs, max_blocks_per_seq]
    context_lens  : int32 [num_seqs]

Token position p of sequence s lives in physical block
``block_tables[s, p // block_size]`` at slot ``p % block_size`` (glossary
entry, "PagedAttentionの解決策": the block table maps logical blocks to
physical blocks, which need not be contiguous).

Readings where the pages are silent:
* GQA (glossary entry, "他のKVキャッシュ最適化との組み合わせ", only names
  GQA): query head h reads KV head ``h // (num_q_heads // num_kv_heads)``.
* A sequence with context length 0 is a padding slot: its output is zeros.
"""

import numpy as np

from .numerics import to_f64

BLOCK_SIZE = 16


def gather_kv(pool_f64, table_row, length, kv_head, block_size=BLOCK_SIZE, start=0):
    """Contiguous [length - start, head_dim] copy of positions start .. length-1
    of one sequence's K (or V) for one KV head.

    Position p is read from physical block table_row[p // block_size],
    slot p % block_size.
    """
    head_dim = pool_f64.shape[-1]
    out = np.empty((length - start, head_dim), dtype=np.float64)
    for p in range(start, length):
        block = int(table_row[p // block_size])
        if block < 0:
            raise ValueError(f"position {p} maps to no block (table entry {block})")
        out[p - start] = pool_f64[block, kv_head, p % block_size]
    return out


def attend(q_vec, K, V, scale):
    """Single-query softmax attention in float64.

    z_p = scale * <q, K_p>;  w = exp(z - max z) / sum exp(z - max z);
    out = sum_p w_p V_p.  Subtracting the maximum does not change w; it only
    keeps exp() in range.
    """
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64)
    z = scale * (K @ q_vec)
    e = np.exp(z - z.max())
    w = e / e.sum()
    return w @ V


def paged_attention_decode(q, k_pool, v_pool, block_tables, context_lens, scale,
                           num_kv_heads, dtype, block_size=BLOCK_SIZE,
                           pairs=None):
    """Reference output, float64 [num_seqs, num_q_heads, head_dim].

    ``q``, ``k_pool`` and ``v_pool`` are fp16 arrays or bf16 bit patterns
    (uint16), per ``dtype``. ``pairs``, when given, restricts the work to a
    list of (seq, q_head) pairs and the result to those rows (other rows are
    NaN); this is how the full-size parity tests sample outputs.
    """
    qf = to_f64(q, dtype)
    num_seqs, num_q_heads, head_dim = qf.shape
    if num_q_heads % num_kv_heads != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = num_q_heads // num_kv_heads
    kf = to_f64(k_pool, dtype)
    vf = to_f64(v_pool, dtype)
    out = np.full((num_seqs, num_q_heads, head_dim), np.nan if pairs is not None else 0.0)
    todo = pairs if pairs is not None else [(s, h) for s in range(num_seqs)
                                            for h in range(num_q_heads)]
    cache = {}
    for s, h in todo:
        g = h // group
        L = int(context_lens[s])
        key = (s, g)
        if key not in cache:
            cache[key] = (gather_kv(kf, block_tables[s], L, g, block_size),
                          gather_kv(vf, block_tables[s], L, g, block_size))
        K, V = cache[key]
        out[s, h] = attend(qf[s, h], K, V, scale)
    return out


def partition_partials(q_vec, K, V, scale, partition_size):
    """Per-partition softmax pieces of one (sequence, head), float64.

    For partition j covering positions [j*P, (j+1)*P):
        m_j = max z over the partition,
        l_j = sum exp(z - m_j),
        o_j = sum exp(z - m_j) V_p      (not divided by l_j).
    These are the quantities a split-K decode writes before its merge.
    """
    z = scale * (K @ q_vec)
    parts = []
    for start in range(0, K.shape[0], partition_size):
        zj = z[start:start + partition_size]
        m = zj.max()
        e = np.exp(zj - m)
        parts.append((m, e.sum(), e @ V[start:start + partition_size]))
    return parts


def lse_merge(parts):
    """Log-sum-exp merge of partition pieces into the normalised output.

    M = max_j m_j;  out = sum_j e^{m_j - M} o_j / sum_j e^{m_j - M} l_j.
    Because every piece was taken relative to its own maximum, rescaling by
    e^{m_j - M} puts all pieces relative to the global maximum, which is the
    unsplit softmax exactly (up to rounding).
    """
    M = max(m for m, _, _ in parts)
    num = sum(np.exp(m - M) * o for m, _, o in parts)
    den = sum(np.exp(m - M) * l for m, l, _ in parts)
    return num / den


def window_start(length, window):
    """First position a query at position length-1 attends to under a sliding
    window of `window` tokens (the query's own token included); 0 when the
    window is 0 (no window) or covers the whole sequence."""
    if window > 0 and length > window:
        return length - window
    return 0


def paged_attention_decode_window(q, k_pool, v_pool, block_tables, context_lens, scale,
                                  num_kv_heads, dtype, window, block_size=BLOCK_SIZE):
    """Sliding-window decode: each sequence's query attends over its last
    `window` tokens only, positions window_start(L, window) .. L-1 (glossary
    entry "PagedAttention（ページドアテンション）", section
    "他のKVキャッシュ最適化との組み合わせ": sliding-window attention combined
    with paging). Block-table entries of blocks wholly before that range are
    never read. float64 [num_seqs, num_q_heads, head_dim]."""
    qf = to_f64(q, dtype)
    num_seqs, num_q_heads, head_dim = qf.shape
    group = num_q_heads // num_kv_heads
    kf = to_f64(k_pool, dtype)
    vf = to_f64(v_pool, dtype)
    out = np.zeros((num_seqs, num_q_heads, head_dim))
    for s in range(num_seqs):
        L = int(context_lens[s])
        start = window_start(L, window)
        for g in range(num_kv_heads):
            K = gather_kv(kf, block_tables[s], L, g, block_size, start)
            V = gather_kv(vf, block_tables[s], L, g, block_size, start)
            for h in range(g * group, (g + 1) * group):
                out[s, h] = attend(qf[s, h], K, V, scale)
    return out
