"""Pins of the oracle block manager: the pages' worked example, a hand-derived
copy-on-write trace, the last-block waste bound, conservation of blocks, and
transactional failure."""

import json
import os

import numpy as np
import pytest

from oracle import attention as OA
from oracle import cache_ops as OC
from oracle.block_manager import OracleBlockManager, OutOfBlocks, InvalidArgument

BS = 16


def test_glossary_100_token_example(golden_dir):
    with open(os.path.join(golden_dir, "block_table_example.json")) as f:
        ex = json.load(f)
    bm = OracleBlockManager(ex["num_blocks"], initial_free_order=ex["initial_free_order"])
    bm.add_seq("A", ex["num_tokens"])
    table = bm.block_table("A")
    assert table == ex["expected_table"]
    assert table[:3] == [3, 7, 1]
    in_last = ex["num_tokens"] - (len(table) - 1) * BS
    assert in_last == ex["expected_tokens_in_last_block"]
    assert len(table) * BS - ex["num_tokens"] == ex["expected_unused_slots"]
    assert bm.num_free() == ex["expected_num_free_after_add"]


def test_cow_n3_trace(golden_dir):
    with open(os.path.join(golden_dir, "cow_n3_example.json")) as f:
        ex = json.load(f)
    bm = OracleBlockManager(ex["num_blocks"], initial_free_order=ex["initial_free_order"])
    bm.add_seq(0, ex["prompt_tokens"])
    for c in ex["children"]:
        bm.fork(0, c)
    for step in ex["expected_appends"]:
        assert bm.append_slot(step["seq"]) == (step["slot"], step["cow_src"], step["cow_dst"])
    for s, t in ex["expected_tables_after_appends"].items():
        assert bm.block_table(int(s)) == t
    for b, r in ex["expected_refcounts_after_appends"].items():
        assert bm.refcount[int(b)] == r
    assert bm.num_free() == ex["expected_num_free_after_appends"]
    for s in [0] + ex["children"]:
        bm.free_seq(s)
    assert bm.free == ex["expected_free_stack_after_all_freed"]


def test_prompt_multiple_of_16_needs_no_copy():
    bm = OracleBlockManager(10)
    bm.add_seq(0, 32)
    bm.fork(0, 1)
    bm.fork(0, 2)
    for s in range(3):
        slot, src, dst = bm.append_slot(s)
        assert (src, dst) == (-1, -1)
        assert slot % BS == 0                                  # first slot of a fresh block
    assert bm.refcount[bm.block_table(0)[0]] == 3              # full prompt blocks stay shared


def _check_invariants(bm):
    ref = [0] * bm.num_blocks
    for s, t in bm.tables.items():
        L = bm.lengths[s]
        assert len(t) == -(-L // BS)
        assert len(t) * BS - L <= 15                           # waste only in the last block
        for b in t:
            ref[b] += 1
    assert ref == bm.refcount
    referenced = sum(1 for r in ref if r > 0)
    assert referenced + bm.num_free() == bm.num_blocks
    assert len(set(bm.free)) == len(bm.free)
    assert all(bm.refcount[b] == 0 for b in bm.free)


def test_random_trace_invariants():
    rng = np.random.default_rng(0)
    bm = OracleBlockManager(200, initial_free_order=rng.permutation(200))
    live, nxt = [], 0
    for _ in range(3000):
        op = rng.integers(0, 10)
        try:
            if op < 2 or not live:
                bm.add_seq(nxt, int(rng.integers(0, 60)))
                live.append(nxt)
                nxt += 1
            elif op < 3:
                bm.fork(live[int(rng.integers(len(live)))], nxt)
                live.append(nxt)
                nxt += 1
            elif op < 4:
                bm.free_seq(live.pop(int(rng.integers(len(live)))))
            else:
                bm.append_slot(live[int(rng.integers(len(live)))])
        except OutOfBlocks:
            pass
        _check_invariants(bm)
    for s in list(live):
        bm.free_seq(s)
    assert bm.num_free() == 200 and all(r == 0 for r in bm.refcount)


def _state(bm):
    return (list(bm.free), list(bm.refcount), {k: list(v) for k, v in bm.tables.items()},
            dict(bm.lengths))


def test_failures_leave_state_unchanged():
    bm = OracleBlockManager(2, initial_free_order=[0, 1])
    bm.add_seq(0, 5)                                            # takes block 1
    bm.fork(0, 1)
    bm.fork(0, 2)
    snap = _state(bm)
    with pytest.raises(OutOfBlocks):
        bm.add_seq(3, 17)                                       # needs 2 blocks, 1 free
    assert _state(bm) == snap
    assert bm.append_slot(0) == (0 * BS + 5, 1, 0)              # copy-on-write takes block 0
    snap = _state(bm)
    with pytest.raises(OutOfBlocks):
        bm.append_slot(1)                                       # block 1 still shared, none free
    assert _state(bm) == snap
    bm2 = OracleBlockManager(1)
    bm2.add_seq(0, 16)
    snap2 = _state(bm2)
    with pytest.raises(OutOfBlocks):
        bm2.append_slot(0)                                      # full last block, none free
    assert _state(bm2) == snap2
    with pytest.raises(InvalidArgument):
        bm.free_seq(42)
    with pytest.raises(InvalidArgument):
        bm.fork(0, 1)
    with pytest.raises(InvalidArgument):
        bm.add_seq(0, 3)
    assert _state(bm) == snap


def test_cow_siblings_share_prefix_outputs():
    """Siblings with the same query over the shared prompt give identical outputs;
    after copy-on-write the copied block's written slots equal the source's."""
    rng = np.random.default_rng(3)
    hkv, d, prompt, n = 2, 8, 37, 4
    bm = OracleBlockManager(40, initial_free_order=rng.permutation(40))
    bm.add_seq(0, prompt)
    for c in range(1, n):
        bm.fork(0, c)
    kp = rng.standard_normal((40, hkv, BS, d)).astype(np.float16)
    vp = rng.standard_normal((40, hkv, BS, d)).astype(np.float16)
    pairs, slots = [], []
    for s in range(n):
        slot, src, dst = bm.append_slot(s)
        slots.append(slot)
        if src >= 0:
            pairs.append((src, dst))
    assert len(pairs) == n - 1
    kp, vp = OC.copy_blocks(kp, vp, np.array(pairs, np.int64))
    for src, dst in pairs:
        assert np.array_equal(kp[dst, :, :prompt % BS], kp[src, :, :prompt % BS])
    newk = rng.standard_normal((n, hkv, d)).astype(np.float16)
    kp, vp = OC.reshape_and_cache(newk, newk, kp, vp, np.array(slots, np.int64))
    q = np.repeat(rng.standard_normal((1, hkv, d)).astype(np.float16), n, axis=0)
    rows, _ = bm.padded_tables(list(range(n)), 4)
    tables = np.array(rows, np.int32)
    shared = OA.paged_attention_decode(q, kp, vp, tables, np.full(n, prompt, np.int32), 0.3, hkv, "f16")
    for s in range(1, n):
        assert np.array_equal(shared[s], shared[0])
    grown = OA.paged_attention_decode(q, kp, vp, tables, np.full(n, prompt + 1, np.int32), 0.3, hkv, "f16")
    assert not np.array_equal(grown[1], grown[0])              # tails diverge after the write


# ---- beam search and shared prefixes -------------------------------------------
def _beam_golden(golden_dir):
    import json as _json
    with open(os.path.join(golden_dir, "beam_prefix_example.json")) as f:
        return _json.load(f)


def _check_refcounts(bm):
    """Every block's refcount equals the number of live table entries naming it;
    a block is free exactly when its refcount is 0."""
    counts = [0] * bm.num_blocks
    for t in bm.tables.values():
        for b in t:
            if b >= 0:
                counts[b] += 1
    assert counts == bm.refcount
    assert sorted(bm.free) == [b for b in range(bm.num_blocks) if counts[b] == 0]


def test_beam_step_golden(golden_dir):
    ex = _beam_golden(golden_dir)
    g = ex["beam"]
    bm = OracleBlockManager(ex["num_blocks"])
    bm.add_seq(0, g["prompt_tokens"])
    bm.fork(0, 1)
    bm.fork(0, 2)
    res = [bm.append_slot(s) for s in (0, 1, 2)]
    assert [r[0] for r in res] == g["first_append_slots"]
    assert [[r[1], r[2]] for r in res if r[1] >= 0] == g["first_pairs"]
    bm.beam_reorder(g["old_ids"], g["parents"], g["new_ids"])
    assert {str(k): v for k, v in bm.tables.items()} == g["tables_after_reorder"]
    for b, r in g["refcounts_after_reorder"].items():
        assert bm.refcount[int(b)] == r
    assert bm.free == g["free_after_reorder"]
    res = [bm.append_slot(s) for s in g["new_ids"]]
    assert [r[0] for r in res] == g["second_append_slots"]
    assert [[r[1], r[2]] for r in res if r[1] >= 0] == g["second_pairs"]
    _check_refcounts(bm)


def test_prefix_sharing_golden(golden_dir):
    ex = _beam_golden(golden_dir)
    g = ex["prefix"]
    bm = OracleBlockManager(ex["num_blocks"])
    bm.add_seq(1, g["donor_tokens"])
    assert bm.block_table(1) == g["donor_table"]
    assert bm.add_seq_with_prefix(2, g["num_tokens"], 1, g["prefix_tokens"]) == g["shared_tokens"]
    assert bm.block_table(2) == g["table"]
    bm.free_seq(1)
    assert bm.free == g["free_after_donor_freed"]
    _check_refcounts(bm)


def test_prefix_sharing_is_block_granular():
    bm = OracleBlockManager(16)
    bm.add_seq(1, 37)                                    # blocks 15, 14, 13
    assert bm.add_seq_with_prefix(2, 100, 1, 31) == 16   # only one whole block in 31 tokens
    assert bm.block_table(2)[0] == 15 and bm.refcount[14] == 1
    assert bm.add_seq_with_prefix(3, 20, 1, 37) == 16    # capped by the new request's 20 tokens
    assert bm.add_seq_with_prefix(4, 5, 1, 37) == 0      # shorter than a block: nothing shared
    assert bm.add_seq_with_prefix(5, 64, 1, 64) == 32    # capped by the donor's 37 tokens
    _check_refcounts(bm)
    # a shared prefix block is copied on write like any shared block
    bm.free_seq(2)
    bm.free_seq(3)
    bm.free_seq(4)
    bm.free_seq(5)
    _check_refcounts(bm)
    assert bm.refcount[15] == 1


def test_prefix_sharing_failures_leave_state_unchanged():
    bm = OracleBlockManager(4)
    bm.add_seq(1, 40)                                    # 3 blocks, 1 free
    before = (list(bm.free), list(bm.refcount), {k: list(v) for k, v in bm.tables.items()})
    with pytest.raises(OutOfBlocks):
        bm.add_seq_with_prefix(2, 80, 1, 40)             # needs 5 - 2 = 3 fresh
    with pytest.raises(InvalidArgument):
        bm.add_seq_with_prefix(1, 10, 1, 10)             # id exists
    with pytest.raises(InvalidArgument):
        bm.add_seq_with_prefix(3, 10, 9, 10)             # unknown donor
    assert (bm.free, bm.refcount, bm.tables) == before
    bm.release_before(1, 16)
    with pytest.raises(InvalidArgument):
        bm.add_seq_with_prefix(3, 40, 1, 40)             # donor released its first block
    assert 3 not in bm.tables and bm.tables[1][0] == -1
    _check_refcounts(bm)


def test_beam_reorder_rules():
    bm = OracleBlockManager(32)
    bm.add_seq(0, 33)
    for c in (1, 2, 3):
        bm.fork(0, c)
    for s in range(4):
        bm.append_slot(s)
    # ids may be reused; beams that no one continues free their private blocks
    bm.beam_reorder([0, 1, 2, 3], [3, 3, 0, 1], [0, 1, 2, 3])
    assert bm.block_table(0) == bm.block_table(1)
    _check_refcounts(bm)
    free_before = bm.num_free()
    with pytest.raises(InvalidArgument):
        bm.beam_reorder([0, 1], [0, 2], [5, 6])          # parent index out of range
    with pytest.raises(InvalidArgument):
        bm.beam_reorder([0, 1], [0, 1], [5, 5])          # duplicate new ids
    with pytest.raises(InvalidArgument):
        bm.beam_reorder([0, 1], [0, 1], [2, 6])          # 2 is a live sequence outside old_ids
    with pytest.raises(InvalidArgument):
        bm.beam_reorder([0, 0], [0, 1], [5, 6])          # duplicate old ids
    assert bm.num_free() == free_before
    # multi-level: beams of beams, then everything is returned
    for step in range(40):
        olds = sorted(bm.tables)
        rng = np.random.default_rng(step)
        parents = rng.integers(0, len(olds), 4).tolist()
        news = [100 * (step + 1) + i for i in range(4)]
        bm.beam_reorder(olds, parents, news)
        for n in news:
            bm.append_slot(n)
        _check_refcounts(bm)
    for s in list(bm.tables):
        bm.free_seq(s)
    assert sorted(bm.free) == list(range(32))
