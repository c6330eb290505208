"""Pins of the oracle's memory-utilisation simulation: hand-worked traces
(tests/golden/memsim_traces.json), closed forms with ample capacity, and
invariants under memory pressure."""

import json
import os

import numpy as np
import pytest

import oracle.memsim as OM

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "memsim_traces.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_worked_traces(case):
    P, O = zip(*case["requests"])
    r = OM.simulate(P, O, case["num_blocks"], case["scheme"], case["max_len"], case["max_new_tokens"])
    assert [list(x) for x in r["records"]] == case["records"]
    for key in ("completed", "rejected", "preemptions", "fragmentation_stalls", "useful_tokens"):
        assert r[key] == case[key], key


def _random_trace(rng, n, pmax, omax):
    return rng.integers(1, pmax + 1, n).tolist(), rng.integers(1, omax + 1, n).tolist()


@pytest.mark.parametrize("seed", range(4))
def test_ample_capacity_closed_forms(seed):
    # every request fits at once: all admitted at step 0, request i holds
    # P_i + t + 1 tokens after decode t for t < O_i
    rng = np.random.default_rng(seed)
    P, O = _random_trace(rng, 12, 60, 40)
    max_len = 128
    nb = 12 * max_len // 16
    steps = max(O)
    c = OM.simulate(P, O, nb, "contiguous", max_len)
    p = OM.simulate(P, O, nb, "paged", max_len)
    for r in (c, p):
        assert r["steps"] == steps and r["completed"] == 12 and r["preemptions"] == 0
        assert r["useful_tokens"] == sum(O)
    for t in range(steps):
        live = [i for i in range(12) if O[i] > t]
        stored = sum(P[i] + t + 1 for i in live)
        assert c["records"][t] == (len(live), stored, len(live) * max_len)
        paged_alloc = sum(16 * ((P[i] + t + 1 + 15) // 16) for i in live)
        assert p["records"][t] == (len(live), stored, paged_alloc)
    # utilisation of the reserved memory, closed form
    used = sum(o * p_ + o * (o + 1) // 2 for p_, o in zip(P, O))
    assert sum(x[1] for x in c["records"]) == used
    assert sum(x[2] for x in c["records"]) == max_len * sum(O)


@pytest.mark.parametrize("scheme", ["paged", "contiguous"])
@pytest.mark.parametrize("seed", range(6))
def test_invariants_under_pressure(scheme, seed):
    rng = np.random.default_rng(100 + seed)
    P, O = _random_trace(rng, 40, 70, 50)
    nb, max_len = 24, 128
    r = OM.simulate(P, O, nb, scheme, max_len, max_new_tokens=int(rng.integers(50, 100)))
    cap = nb * 16
    assert r["completed"] + r["rejected"] == 40
    for running, stored, alloc in r["records"]:
        assert 0 < running and stored <= alloc <= cap
        if scheme == "paged":
            assert alloc - stored <= 15 * running      # waste only in each sequence's last block
    if scheme == "paged":
        assert r["preemptions"] > 0                    # the pool is too small to avoid it
        assert r["rejected"] == 0


def test_equal_reservations_never_fragment():
    # every request reserves max_len: the arena holds exactly cap // max_len of them
    rng = np.random.default_rng(9)
    P, O = _random_trace(rng, 30, 50, 60)
    r = OM.simulate(P, O, 40, "contiguous", 128)   # 640 slots = 5 reservations
    assert r["fragmentation_stalls"] == 0
    assert max(x[0] for x in r["records"]) == 5
    assert all(x[2] == 128 * x[0] for x in r["records"])


def test_first_free_run():
    used = [True, False, False, True, False, False, False]
    assert OM.first_free_run(used, 2) == 1
    assert OM.first_free_run(used, 3) == 4
    assert OM.first_free_run(used, 4) is None
