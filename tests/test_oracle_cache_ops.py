"""Pins of the reshape_and_cache and copy_blocks oracles.

Both are pure copies, so they are pinned by exact element checks written with
independent indexing, by "gather after write" (the new token is the last
position of its sequence), and by snapshot semantics for copy_blocks.
"""

import numpy as np

from oracle import attention as OA
from oracle import cache_ops as OC
from oracle.block_manager import OracleBlockManager

BS = 16


def _pools(nb, hkv, d, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 16, size=(2, nb, hkv, BS, d), dtype=np.uint16)
    return bits[0], bits[1]


def test_reshape_writes_exactly_the_slots_and_nothing_else():
    nb, hkv, d = 6, 3, 8
    kp, vp = _pools(nb, hkv, d, 0)
    rng = np.random.default_rng(1)
    k = rng.integers(0, 2 ** 16, size=(4, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 2 ** 16, size=(4, hkv, d), dtype=np.uint16)
    slots = np.array([0, 95, -1, 37], np.int64)   # block 0 slot 0; block 5 slot 15; skip; block 2 slot 5
    nk, nv = OC.reshape_and_cache(k, v, kp, vp, slots)
    expect_k, expect_v = kp.copy(), vp.copy()
    for t, (b, o) in {0: (0, 0), 1: (5, 15), 3: (2, 5)}.items():
        expect_k[b, :, o, :] = k[t]
        expect_v[b, :, o, :] = v[t]
    assert np.array_equal(nk, expect_k) and np.array_equal(nv, expect_v)
    assert np.array_equal(kp, _pools(nb, hkv, d, 0)[0])        # input untouched


def test_reshape_then_gather_sees_new_token_last():
    # one new token per sequence at its next slot, as a decode step does
    bm = OracleBlockManager(8, initial_free_order=list(range(8)))
    lengths = [5, 16, 33]
    for s, L in enumerate(lengths):
        bm.add_seq(s, L)
    slots = [bm.append_slot(s)[0] for s in range(3)]
    d = 4
    kp = np.zeros((8, 1, BS, d), np.float16)
    vp = np.zeros((8, 1, BS, d), np.float16)
    newk = np.arange(3 * d, dtype=np.float16).reshape(3, 1, d) + 1
    nk, nv = OC.reshape_and_cache(newk, -newk, kp, vp, np.array(slots, np.int64))
    kf = nk.astype(np.float64)
    for s, L in enumerate(lengths):
        K = OA.gather_kv(kf, bm.block_table(s), L + 1, 0)
        assert np.array_equal(K[L], newk[s, 0].astype(np.float64))
        assert np.all(K[:L] == 0)


def test_copy_blocks_copies_whole_blocks_from_a_snapshot():
    nb, hkv, d = 6, 2, 4
    kp, vp = _pools(nb, hkv, d, 2)
    nk, nv = OC.copy_blocks(kp, vp, np.array([[1, 4], [3, 5]], np.int64))
    for b in range(nb):
        src = {4: 1, 5: 3}.get(b, b)
        assert np.array_equal(nk[b], kp[src]) and np.array_equal(nv[b], vp[src])
    # a chain (0->1, 1->2) reads block 1 before it is overwritten
    ck, _ = OC.copy_blocks(kp, vp, np.array([[1, 2], [0, 1]], np.int64))
    assert np.array_equal(ck[2], kp[1]) and np.array_equal(ck[1], kp[0])
    # empty pair list is the identity
    ek, ev = OC.copy_blocks(kp, vp, np.zeros((0, 2), np.int64))
    assert np.array_equal(ek, kp) and np.array_equal(ev, vp)
