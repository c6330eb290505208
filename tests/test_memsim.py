"""The product's memory-utilisation simulator (C++ block manager, free-span
arena) against the oracle's model: identical step records and counters."""

import json
import os

import numpy as np
import pytest

import oracle.memsim as OM
from paged_kv_cache_217_gb300 import memsim as MS
from paged_kv_cache_217_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "memsim_traces.json")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_217_gb300 import build
    build.build()


def _same(prod, orc):
    assert [(x.running, x.stored_tokens, x.allocated_slots) for x in prod.records] == \
        [tuple(x) for x in orc["records"]]
    assert prod.steps == orc["steps"]
    for key in ("completed", "rejected", "preemptions", "fragmentation_stalls", "generated_tokens",
                "useful_tokens"):
        assert getattr(prod, key) == orc[key], key


def test_golden_traces():
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        P, O = zip(*c["requests"])
        args = (P, O, c["num_blocks"], c["scheme"], c["max_len"], c["max_new_tokens"])
        _same(MS.simulate(*args), OM.simulate(*args))


@pytest.mark.parametrize("scheme", ["paged", "contiguous"])
@pytest.mark.parametrize("seed", range(5))
def test_random_traces_match_oracle(scheme, seed):
    rng = np.random.default_rng(seed)
    n = 60
    P = rng.integers(1, 90, n).tolist()
    O = rng.integers(1, 70, n).tolist()
    nb = int(rng.integers(20, 60))
    order = W.shuffled_free_order(nb, seed)
    args = (P, O, nb, scheme, 160, int(rng.integers(40, 200)))
    _same(MS.simulate(*args, free_order=order), OM.simulate(*args, free_order=order))


@pytest.mark.parametrize("trace", ["llama13b", "llama3_8b"])
def test_layer_length_traces_match_oracle(trace):
    P, O, max_len = W.memsim_trace(trace, 48, seed=3)
    nb = 6 * max_len // 16
    for scheme in ("paged", "contiguous"):
        _same(MS.simulate(P, O, nb, scheme, max_len), OM.simulate(P, O, nb, scheme, max_len))


def test_paged_waste_below_four_percent():
    # the pages: waste only in the last block, under 4 % of the KV memory
    P, O, max_len = W.memsim_trace("llama13b", 256, seed=0)
    r = MS.simulate(P, O, 16 * max_len // 16, "paged", max_len)
    c = MS.simulate(P, O, 16 * max_len // 16, "contiguous", max_len)
    assert r.utilisation_of_allocated > 0.96
    assert c.utilisation_of_allocated < 0.5
    assert r.tokens_per_step > 1.5 * c.tokens_per_step


def test_rejects_bad_traces():
    with pytest.raises(ValueError):
        MS.simulate([5], [0], 4, "paged", 64)
    with pytest.raises(ValueError):
        MS.simulate([5], [1], 4, "buddy", 64)
