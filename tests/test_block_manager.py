"""The C++ block manager (through the C ABI) against the oracle block manager:
bit-exact tables, slots, copy-on-write pairs, refcounts and free stacks on
scripted traces; transactional failure; host-side pair checks. CPU only."""

import json
import os

import numpy as np
import pytest

from oracle.block_manager import OracleBlockManager, OutOfBlocks as OracleOOB, InvalidArgument
from paged_kv_cache_217_gb300 import binding as B
from paged_kv_cache_217_gb300 import workloads as W

BS = 16


def _same_state(cbm, obm, seq_ids):
    assert cbm.free_stack() == obm.free
    assert [cbm.refcount(b) for b in range(obm.num_blocks)] == obm.refcount
    assert cbm.num_seqs() == len(obm.tables)
    for s in seq_ids:
        assert cbm.block_table(s) == obm.block_table(s)
        assert cbm.seq_len(s) == obm.length(s)


def test_glossary_example_and_cow_trace(golden_dir):
    with open(os.path.join(golden_dir, "block_table_example.json")) as f:
        ex = json.load(f)
    bm = B.BlockManager(ex["num_blocks"], ex["initial_free_order"])
    bm.add_seq(1, ex["num_tokens"])
    assert bm.block_table(1) == ex["expected_table"]
    assert bm.num_free() == ex["expected_num_free_after_add"]

    with open(os.path.join(golden_dir, "cow_n3_example.json")) as f:
        ex = json.load(f)
    bm = B.BlockManager(ex["num_blocks"], ex["initial_free_order"])
    bm.add_seq(0, ex["prompt_tokens"])
    for c in ex["children"]:
        bm.fork(0, c)
    for step in ex["expected_appends"]:
        assert bm.append_slot(step["seq"]) == (step["slot"], step["cow_src"], step["cow_dst"])
    for s, t in ex["expected_tables_after_appends"].items():
        assert bm.block_table(int(s)) == t
    for b, r in ex["expected_refcounts_after_appends"].items():
        assert bm.refcount(int(b)) == r
    for s in [0] + ex["children"]:
        bm.free_seq(s)
    assert bm.free_stack() == ex["expected_free_stack_after_all_freed"]


def test_tiny_decode_tables_match_oracle():
    shape = W.tiny_decode()
    order = W.shuffled_free_order(64, 0)
    cbm, obm = B.BlockManager(64, order), OracleBlockManager(64, initial_free_order=order)
    for s, L in enumerate(shape.context_lens.tolist()):
        cbm.add_seq(s, L)
        obm.add_seq(s, L)
    _same_state(cbm, obm, range(4))
    slots, pairs = cbm.append_slots(range(4))
    want = [obm.append_slot(s) for s in range(4)]
    assert slots.tolist() == [w[0] for w in want] and pairs.shape == (0, 2)
    _same_state(cbm, obm, range(4))
    t, lens = cbm.block_tables(range(4), 5)
    rows, olens = obm.padded_tables(range(4), 5)
    assert t.tolist() == rows and lens.tolist() == olens


@pytest.mark.parametrize("seed", [0, 1])
def test_parallel_sampling_trace_matches_oracle(seed):
    trace = W.opt66b_parallel_sampling(seed)
    nb = trace.block_budget()
    order = W.shuffled_free_order(nb, seed)
    cbm, obm = B.BlockManager(nb, order), OracleBlockManager(nb, initial_free_order=order)
    cplan = W.drive_parallel_sampling(trace, cbm)
    oplan = W.drive_parallel_sampling(trace, obm)
    assert cplan.pairs == oplan.pairs
    assert len(cplan.step_slots) == len(oplan.step_slots)
    for (ca, cs), (oa, os_) in zip(cplan.step_slots, oplan.step_slots):
        assert ca == oa and np.array_equal(cs, os_)
    _same_state(cbm, obm, cplan.seq_ids)
    # refcount-driven copy-on-write: n-1 copies per prompt whose last block is
    # partial and whose samples all append; none for prompts of 16k tokens
    expect = 0
    for i, plen in enumerate(trace.prompt_lens.tolist()):
        writers = int((trace.tail_lens[i] > 0).sum())
        if plen % BS:
            expect += writers if writers < trace.n else trace.n - 1
    assert len(cplan.pairs) == expect
    B.check_copy_pairs(cplan.pairs, nb)
    for sid in cplan.seq_ids:
        L = cplan.final_lens[sid]
        assert cbm.seq_len(sid) == L
        assert len(cbm.block_table(sid)) * BS - L <= 15


def test_random_trace_matches_oracle():
    rng = np.random.default_rng(11)
    nb = 150
    order = rng.permutation(nb)
    cbm, obm = B.BlockManager(nb, order), OracleBlockManager(nb, initial_free_order=order)
    live, nxt = [], 0
    for it in range(2500):
        op = int(rng.integers(0, 12))
        if op >= 10 and live:             # sliding-window release
            sid = live[int(rng.integers(len(live)))]
            first = int(rng.integers(0, obm.length(sid) + 1))
            assert cbm.release_before(sid, first) == obm.release_before(sid, first)
            continue
        if op < 2 or not live:
            args, ops = (nxt, int(rng.integers(0, 70))), ("add_seq", "add_seq")
        elif op < 3:
            args, ops = (live[int(rng.integers(len(live)))], nxt), ("fork", "fork")
        elif op < 4:
            args, ops = (live[int(rng.integers(len(live)))],), ("free_seq", "free_seq")
        else:
            args, ops = (live[int(rng.integers(len(live)))],), ("append_slot", "append_slot")
        c_exc = o_exc = None
        try:
            cres = getattr(cbm, ops[0])(*args)
        except B.OutOfBlocks as e:
            c_exc = e
        try:
            ores = getattr(obm, ops[1])(*args)
        except OracleOOB as e:
            o_exc = e
        assert (c_exc is None) == (o_exc is None), f"step {it}: {ops[0]}{args}"
        if c_exc is None:
            assert cres == ores
            if ops[0] in ("add_seq", "fork"):
                live.append(nxt)
                nxt += 1
            elif ops[0] == "free_seq":
                live.remove(args[0])
        if it % 50 == 0:
            _same_state(cbm, obm, live)
    _same_state(cbm, obm, live)


def test_batch_append_is_all_or_nothing():
    bm = B.BlockManager(3, [0, 1, 2])
    bm.add_seq(0, 16)
    bm.add_seq(1, 16)
    bm.add_seq(2, 0)              # empty sequence, no block yet
    before = (bm.free_stack(), [bm.refcount(b) for b in range(3)],
              [bm.block_table(s) for s in range(3)], [bm.seq_len(s) for s in range(3)])
    with pytest.raises(B.OutOfBlocks):
        bm.append_slots([0, 1, 2])    # three fresh blocks needed, one free
    after = (bm.free_stack(), [bm.refcount(b) for b in range(3)],
             [bm.block_table(s) for s in range(3)], [bm.seq_len(s) for s in range(3)])
    assert before == after
    # copy-on-write inside a failing batch is undone too
    bm = B.BlockManager(3, [0, 1, 2])
    bm.add_seq(0, 5)
    bm.fork(0, 1)
    bm.fork(0, 2)
    before = (bm.free_stack(), [bm.refcount(b) for b in range(3)], [bm.block_table(s) for s in range(3)])
    with pytest.raises(B.OutOfBlocks):
        bm.append_slots([0, 1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0])
    assert before == (bm.free_stack(), [bm.refcount(b) for b in range(3)],
                      [bm.block_table(s) for s in range(3)])
    slots, pairs = bm.append_slots([0, 1, 2])
    assert pairs.tolist() == [[2, 1], [2, 0]] and slots.tolist() == [21, 5, 37]


def test_invalid_arguments():
    with pytest.raises(B.PagedKVError):
        B.BlockManager(4, [0, 1, 1, 2])
    with pytest.raises(B.PagedKVError):
        B.BlockManager(4, block_size=8)
    bm = B.BlockManager(4)
    with pytest.raises(B.PagedKVError):
        bm.free_seq(3)
    bm.add_seq(3, 1)
    with pytest.raises(B.PagedKVError):
        bm.add_seq(3, 1)
    with pytest.raises(B.PagedKVError):
        bm.fork(9, 10)
    with pytest.raises(B.PagedKVError):
        bm.block_tables([3], 0)
    with pytest.raises(InvalidArgument):
        OracleBlockManager(4).fork(9, 10)


def test_check_copy_pairs():
    B.check_copy_pairs([[1, 2], [1, 3], [4, 5]], 6)       # one src copied twice is fine
    B.check_copy_pairs(np.zeros((0, 2), np.int64), 6)
    for bad in ([[1, 2], [3, 2]], [[1, 2], [2, 3]], [[0, 6]], [[-1, 2]]):
        with pytest.raises(B.PagedKVError):
            B.check_copy_pairs(bad, 6)


def test_release_before_matches_oracle_and_rejects_bad_positions():
    order = list(range(12))
    cbm, obm = B.BlockManager(12, order), OracleBlockManager(12, initial_free_order=order)
    for bm in (cbm, obm):
        bm.add_seq(1, 70)
        bm.fork(1, 2)
    assert cbm.release_before(1, 50) == obm.release_before(1, 50) == 3
    assert cbm.release_before(2, 33) == obm.release_before(2, 33) == 2
    _same_state(cbm, obm, [1, 2])
    for bm in (cbm, obm):
        bm.fork(1, 3)
        bm.append_slot(3)
        bm.free_seq(2)
    _same_state(cbm, obm, [1, 3])
    with pytest.raises(B.PagedKVError):
        cbm.release_before(1, 71)
    with pytest.raises(B.PagedKVError):
        cbm.release_before(7, 0)
    _same_state(cbm, obm, [1, 3])


def test_beam_and_prefix_golden(golden_dir):
    with open(os.path.join(golden_dir, "beam_prefix_example.json")) as f:
        ex = json.load(f)
    g = ex["beam"]
    bm = B.BlockManager(ex["num_blocks"])
    bm.add_seq(0, g["prompt_tokens"])
    bm.fork(0, 1)
    bm.fork(0, 2)
    slots, pairs = bm.append_slots([0, 1, 2])
    assert slots.tolist() == g["first_append_slots"] and pairs.tolist() == g["first_pairs"]
    bm.beam_reorder(g["old_ids"], g["parents"], g["new_ids"])
    for s, t in g["tables_after_reorder"].items():
        assert bm.block_table(int(s)) == t
    for b, r in g["refcounts_after_reorder"].items():
        assert bm.refcount(int(b)) == r
    assert bm.free_stack() == g["free_after_reorder"]
    slots, pairs = bm.append_slots(g["new_ids"])
    assert slots.tolist() == g["second_append_slots"] and pairs.tolist() == g["second_pairs"]

    p = ex["prefix"]
    bm = B.BlockManager(ex["num_blocks"])
    bm.add_seq(1, p["donor_tokens"])
    assert bm.add_seq_with_prefix(2, p["num_tokens"], 1, p["prefix_tokens"]) == p["shared_tokens"]
    assert bm.block_table(2) == p["table"]
    bm.free_seq(1)
    assert bm.free_stack() == p["free_after_donor_freed"]


def test_beam_and_prefix_random_trace_matches_oracle():
    rng = np.random.default_rng(21)
    nb = 200
    order = rng.permutation(nb)
    cbm, obm = B.BlockManager(nb, order), OracleBlockManager(nb, initial_free_order=order)
    live, nxt = [], 0
    for it in range(1500):
        op = int(rng.integers(0, 10))
        c_exc = o_exc = None
        if op < 2 or not live:
            donor = live[int(rng.integers(len(live)))] if live and op == 1 else None
            n, pre = int(rng.integers(0, 90)), int(rng.integers(0, 90))
            calls = (("add_seq_with_prefix", (nxt, n, donor, pre)) if donor is not None
                     else ("add_seq", (nxt, n)))
        elif op < 4:
            k = int(rng.integers(1, min(len(live), 4) + 1))
            olds = [live[i] for i in rng.choice(len(live), k, replace=False)]
            width = int(rng.integers(1, 5))
            parents = rng.integers(0, k, width).tolist()
            news = [nxt + i for i in range(width)]
            calls = ("beam_reorder", (olds, parents, news))
        elif op < 5:
            calls = ("free_seq", (live[int(rng.integers(len(live)))],))
        else:
            calls = ("append_slot", (live[int(rng.integers(len(live)))],))
        name, args = calls
        try:
            cres = getattr(cbm, name)(*args)
        except B.OutOfBlocks as e:
            c_exc = e
        try:
            ores = getattr(obm, name)(*args)
        except OracleOOB as e:
            o_exc = e
        assert (c_exc is None) == (o_exc is None), f"step {it}: {name}{args}"
        if c_exc is None:
            assert cres == ores, f"step {it}: {name}{args}"
            if name in ("add_seq", "add_seq_with_prefix"):
                live.append(nxt)
                nxt += 1
            elif name == "beam_reorder":
                for o in args[0]:
                    live.remove(o)
                live.extend(args[2])
                nxt += len(args[2])
            elif name == "free_seq":
                live.remove(args[0])
        if it % 25 == 0:
            _same_state(cbm, obm, live)
    _same_state(cbm, obm, live)


def test_beam_reorder_rejects_bad_arguments_atomically():
    bm = B.BlockManager(16)
    bm.add_seq(0, 20)
    bm.fork(0, 1)
    before = (bm.free_stack(), [bm.refcount(b) for b in range(16)])
    for olds, parents, news in (([0, 1], [2], [5]), ([0, 1], [0, 1], [7, 7]), ([0, 0], [0], [5]),
                                ([0, 9], [0], [5]), ([0], [0], [1])):
        with pytest.raises(B.PagedKVError):
            bm.beam_reorder(olds, parents, news)
    assert (bm.free_stack(), [bm.refcount(b) for b in range(16)]) == before
    assert bm.num_seqs() == 2
