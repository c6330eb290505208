"""reshape_and_cache and copy_blocks as plain element-wise copies.

Test infrastructure (see the package docstring).

Both operations move bits and do no arithmetic, so the oracle compares
bit-exactly: it works on the raw 16-bit patterns (any NumPy 16-bit dtype)
and returns new arrays, leaving its inputs untouched.

* reshape_and_cache: each decode step writes the new token's K and V into the
  next slot of its sequence's last block ("KV キャッシュマネージャ" in the
  abeam.tech summary: tokens fill the last block; a full block is followed
  by a newly allocated one). ``slot = physical_block * block_size + offset``;
  a negative slot means "skip this token".
* copy_blocks: copy-on-write ("並列サンプリングやビームサーチでの共有":
  a shared block is duplicated only when a write reaches it). Each
  ``(src, dst)`` pair copies all KV heads and all slots of block ``src`` to
  block ``dst`` in both pools.
"""

import numpy as np

BLOCK_SIZE = 16


def reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, block_size=BLOCK_SIZE):
    """Return (new_k_pool, new_v_pool) with token t's rows written at slot_mapping[t].

    k, v          : [num_tokens, num_kv_heads, head_dim]
    k_pool, v_pool: [num_blocks, num_kv_heads, block_size, head_dim]
    """
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        block, offset = divmod(int(slot), block_size)
        for g in range(kp.shape[1]):
            kp[block, g, offset, :] = k[t, g, :]
            vp[block, g, offset, :] = v[t, g, :]
    return kp, vp


def copy_blocks(k_pool, v_pool, pairs):
    """Return (new_k_pool, new_v_pool) after copying each (src, dst) pair.

    All sources are read from a snapshot taken before any write, so the
    result does not depend on the order of the pairs.
    """
    snap_k = np.array(k_pool, copy=True)
    snap_v = np.array(v_pool, copy=True)
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        kp[int(dst)] = snap_k[int(src)]
        vp[int(dst)] = snap_v[int(src)]
    return kp, vp
