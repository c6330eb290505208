"""Pins of the sliding-window oracle (decode over the last W tokens) and of
the block manager's release of blocks before the window."""

import numpy as np
import pytest

import oracle.attention as OA
import oracle.block_manager as OB
from oracle.numerics import to_f64


def _case(lens, hq, hkv, d, seed, dtype="f16"):
    rng = np.random.default_rng(seed)
    nb = sum(-(-L // 16) for L in lens) + 3
    perm = rng.permutation(nb)
    mb = max(-(-L // 16) for L in lens) + 1
    tables = np.full((len(lens), mb), -1, np.int32)
    k = 0
    for s, L in enumerate(lens):
        n = -(-L // 16)
        tables[s, :n] = perm[k:k + n]
        k += n
    kp = rng.standard_normal((nb, hkv, 16, d)).astype(np.float16)
    vp = rng.standard_normal((nb, hkv, 16, d)).astype(np.float16)
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float16)
    return q, kp, vp, tables, np.array(lens, np.int32)


def test_window_covering_everything_is_full_attention():
    q, kp, vp, t, lens = _case([5, 17, 40, 64], 4, 2, 32, 0)
    full = OA.paged_attention_decode(q, kp, vp, t, lens, 0.2, 2, "f16")
    for w in (0, 64, 65, 1000):
        np.testing.assert_array_equal(OA.paged_attention_decode_window(q, kp, vp, t, lens, 0.2, 2, "f16", w), full)


def test_window_of_one_returns_the_last_value_row():
    q, kp, vp, t, lens = _case([5, 17, 40, 64], 4, 4, 16, 1)
    out = OA.paged_attention_decode_window(q, kp, vp, t, lens, 0.3, 4, "f16", 1)
    vf = to_f64(vp, "f16")
    for s, L in enumerate(lens):
        b, off = t[s, (L - 1) // 16], (L - 1) % 16
        for h in range(4):
            np.testing.assert_array_equal(out[s, h], vf[b, h, off])


@pytest.mark.parametrize("w", [1, 7, 16, 23, 33])
def test_window_equals_full_attention_over_the_last_tokens(w):
    # rebuild every sequence as just its last w tokens in a fresh pool, token by
    # token, and run the (separately pinned) full-attention oracle on it
    lens = [3, 16, 17, 50, 64, 81]
    q, kp, vp, t, L = _case(lens, 6, 3, 16, 2)
    want = OA.paged_attention_decode_window(q, kp, vp, t, L, 0.25, 3, "f16", w)
    n_new = [min(x, w) for x in lens]
    nb = sum(-(-n // 16) for n in n_new)
    kp2 = np.zeros((nb, 3, 16, 16), np.float16)
    vp2 = np.zeros_like(kp2)
    t2 = np.full((len(lens), -(-max(n_new) // 16)), -1, np.int32)
    nxt = 0
    for s, x in enumerate(lens):
        n = n_new[s]
        for j in range(-(-n // 16)):
            t2[s, j] = nxt
            nxt += 1
        for i in range(n):
            p = x - n + i                   # old position
            src_b, src_o = t[s, p // 16], p % 16
            kp2[t2[s, i // 16], :, i % 16] = kp[src_b, :, src_o]
            vp2[t2[s, i // 16], :, i % 16] = vp[src_b, :, src_o]
    got = OA.paged_attention_decode(q, kp2, vp2, t2, np.array(n_new, np.int32), 0.25, 3, "f16")
    np.testing.assert_allclose(want, got, rtol=0, atol=1e-15)


def test_tokens_before_the_window_do_not_matter():
    q, kp, vp, t, lens = _case([70], 2, 2, 16, 3)
    w = 20                                   # window starts at position 50
    base = OA.paged_attention_decode_window(q, kp, vp, t, lens, 0.25, 2, "f16", w)
    kp2, vp2 = kp.copy(), vp.copy()
    for p in range(50):                       # scramble every earlier position
        kp2[t[0, p // 16], :, p % 16] = 7.0
        vp2[t[0, p // 16], :, p % 16] = -3.0
    np.testing.assert_array_equal(OA.paged_attention_decode_window(q, kp2, vp2, t, lens, 0.25, 2, "f16", w), base)
    vp2[t[0, 50 // 16], :, 50 % 16] = 5.0     # position 50 is inside the window
    assert not np.array_equal(OA.paged_attention_decode_window(q, kp2, vp2, t, lens, 0.25, 2, "f16", w), base)


def test_released_entries_are_never_read():
    q, kp, vp, t, lens = _case([70, 40], 2, 2, 16, 4)
    w = 21                                   # starts: 49 -> blocks 0..2 released; 19 -> block 0
    base = OA.paged_attention_decode_window(q, kp, vp, t, lens, 0.25, 2, "f16", w)
    t2 = t.copy()
    t2[0, :3] = -1
    t2[1, :1] = -1
    np.testing.assert_array_equal(OA.paged_attention_decode_window(q, kp, vp, t2, lens, 0.25, 2, "f16", w), base)
    t2[0, 3] = -1                            # block 3 holds positions 48..63, in the window
    with pytest.raises(ValueError):
        OA.paged_attention_decode_window(q, kp, vp, t2, lens, 0.25, 2, "f16", w)


def test_window_start():
    assert OA.window_start(100, 0) == 0
    assert OA.window_start(100, 100) == 0
    assert OA.window_start(100, 30) == 70
    assert OA.window_start(1, 1) == 0


def test_release_before_frees_whole_blocks_in_table_order():
    bm = OB.OracleBlockManager(8)             # free stack pops 7, 6, 5, ...
    bm.add_seq(1, 70)                         # blocks [7, 6, 5, 4, 3]
    assert bm.block_table(1) == [7, 6, 5, 4, 3]
    assert bm.release_before(1, 47) == 2      # blocks 0, 1 hold positions 0..31
    assert bm.block_table(1) == [-1, -1, 5, 4, 3]
    assert bm.free == [0, 1, 2, 7, 6]
    assert bm.release_before(1, 47) == 0      # idempotent
    assert bm.release_before(1, 48) == 1
    assert bm.free[-1] == 5
    slot, src, dst = bm.append_slot(1)        # position 70 -> block 3 (index 4), slot 6
    assert (slot, src, dst) == (3 * 16 + 6, -1, -1)
    bm.free_seq(1)
    assert sorted(bm.free) == list(range(8))
    assert all(r == 0 for r in bm.refcount)


def test_release_before_with_shared_blocks():
    bm = OB.OracleBlockManager(8)
    bm.add_seq(1, 40)                         # [7, 6, 5]
    bm.fork(1, 2)
    assert bm.release_before(1, 32) == 2      # refcounts 2 -> 1: nothing returns to the free list
    assert bm.num_free() == 5 and bm.refcount[7] == 1 and bm.refcount[6] == 1
    bm.fork(1, 3)                             # shares only the live block 5
    assert bm.refcount[5] == 3 and bm.refcount[7] == 1
    assert bm.release_before(2, 16) == 1      # seq 2 drops block 7: freed
    assert bm.free[-1] == 7
    for s in (1, 2, 3):
        bm.free_seq(s)
    assert sorted(bm.free) == list(range(8))


def test_release_before_rejects_bad_arguments():
    bm = OB.OracleBlockManager(4)
    bm.add_seq(1, 20)
    with pytest.raises(OB.InvalidArgument):
        bm.release_before(1, 21)
    with pytest.raises(OB.InvalidArgument):
        bm.release_before(9, 0)
