"""Pins of the oracle's prefix-group planner: a hand-worked batch, and the
group invariants on block-manager batches (forks, beams)."""

import json
import os

import numpy as np
import pytest

import oracle.attention as OA
import oracle.cascade as OK
from oracle.block_manager import OracleBlockManager

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "prefix_groups_example.json")


def test_hand_worked_batch():
    with open(GOLDEN) as f:
        ex = json.load(f)
    for c in ex["cases"]:
        groups, prefix = OK.plan_prefix_groups(ex["tables"], ex["lens"], c["max_members"], c["min_shared"])
        assert [list(g) for g in groups] == c["groups"], c
        assert prefix == c["seq_prefix"], c


def _forked_batch(rng, nb=400):
    """Prompts forked into a few samples each, then a few appends per sample."""
    bm = OracleBlockManager(nb, initial_free_order=rng.permutation(nb))
    ids = []
    for p in range(int(rng.integers(3, 7))):
        root = 100 * p
        bm.add_seq(root, int(rng.integers(1, 120)))
        ids.append(root)
        for c in range(1, int(rng.integers(1, 6))):
            bm.fork(root, root + c)
            ids.append(root + c)
    for _ in range(int(rng.integers(0, 40))):
        bm.append_slot(ids[int(rng.integers(len(ids)))])
    mb = max(len(bm.block_table(s)) for s in ids) + 1
    rows, lens = bm.padded_tables(ids, mb)
    return rows, lens


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("max_members,min_shared", [(8, 1), (4, 2), (2, 3)])
def test_group_invariants(seed, max_members, min_shared):
    rows, lens = _forked_batch(np.random.default_rng(seed))
    groups, prefix = OK.plan_prefix_groups(rows, lens, max_members, min_shared)
    covered = []
    for first, count, P in groups:
        assert 2 <= count <= max_members and P >= min_shared
        members = list(range(first, first + count))
        covered += members
        for m in members:
            assert P <= lens[m] // 16
            assert rows[m][:P] == rows[first][:P] and all(b >= 0 for b in rows[m][:P])
            assert prefix[m] == P
        # the group could not take one more member without dropping below min_shared
        nxt = first + count
        if count < max_members and nxt < len(lens):
            c = OK.common_blocks(rows[nxt - 1], lens[nxt - 1], rows[nxt], lens[nxt])
            assert min(P, c) < min_shared
    assert covered == sorted(set(covered))
    for s in range(len(lens)):
        if s not in covered:
            assert prefix[s] == 0


def test_prefix_and_suffix_merge_to_plain_attention():
    # the decomposition the grouped decode relies on, with the planner's P
    rng = np.random.default_rng(3)
    rows, lens = _forked_batch(rng)
    groups, prefix = OK.plan_prefix_groups(rows, lens, 8, 1)
    assert groups
    d = 16
    nb = 400
    kp = rng.standard_normal((nb, 1, 16, d))
    vp = rng.standard_normal((nb, 1, 16, d))
    for s in range(len(lens)):
        L, P = lens[s], prefix[s]
        if L == 0:
            continue
        K = OA.gather_kv(kp, rows[s], L, 0)
        V = OA.gather_kv(vp, rows[s], L, 0)
        q = rng.standard_normal(d)
        want = OA.attend(q, K, V, 0.25)
        if 0 < 16 * P < L:
            parts = []
            for lo, hi in ((0, 16 * P), (16 * P, L)):
                z = 0.25 * (K[lo:hi] @ q)
                m = z.max()
                e = np.exp(z - m)
                parts.append((m, e.sum(), e @ V[lo:hi]))
            np.testing.assert_allclose(OA.lse_merge(parts), want, rtol=1e-12, atol=1e-12)
