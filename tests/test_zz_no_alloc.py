"""The decode entry point that allocates nothing, checked against the oracle.

pkv_paged_attention_decode_noalloc serves callers that cannot allocate device
memory while they decode (an engine whose allocator already holds nearly all
HBM for the KV pool, or host code that must not call cudaMalloc/cudaFree and
risk a device synchronisation). Its scratch -- split-K partials and arrival
counters, the balanced schedule's slots and counters, and the launch order of
batches of 128..1024 sequences -- is one fixed array inside the library that
every call shares. These tests call it through the C ABI several times in a
row, with shapes and schedules (split-K, balanced, one pass with a launch
order, shared prefix) that put different layouts into that array, and compare
every result element by element with the float64 oracle (and with the
workspace-taking entry point) at the attention tolerance of the other GPU
tests, so stale contents left by one call cannot hide in the next.

This file is collected last on purpose: a run that stops at the first failure
has already run every other test when it gets here.
"""

import numpy as np
import pytest
import torch

import helpers as H
from paged_kv_cache_217_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    H.ensure_built()
    B.device_status(clear=True)
    yield


def _noalloc(case, partition):
    got = case.new_out()
    B.paged_attention_decode_noalloc(got, case.q, case.k_pool, case.v_pool, case.tables, case.lens,
                                     case.scale, partition_size=partition)
    torch.cuda.synchronize()
    return H.to_f64(got)


def _with_workspace(case, partition):
    ref = case.new_out()
    B.paged_attention_decode(ref, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             partition_size=partition)
    torch.cuda.synchronize()
    return H.to_f64(ref)


def _check(case, partition, what):
    got = _noalloc(case, partition)
    H.assert_attention_close(got, H.oracle_full(case), f"{what}: against the oracle")
    H.assert_attention_close(got, _with_workspace(case, partition), f"{what}: against the workspace entry")


def test_noalloc_matches_the_oracle_on_calls_in_a_row():
    # 1: long, split contexts (GQA, bf16): partials, (max, sum) pairs and
    #    counters spread over a large part of the scratch
    a = H.make_case([2048, 700, 33, 1, 0, 1500, 517, 16], 32, 8, 128, "bf16", seed=31)
    need_a = B.workspace_size(8, 32, 8, 128, a.tables.shape[1], 64)
    assert 0 < need_a <= B.NOALLOC_SCRATCH_BYTES
    _check(a, 64, "call 1 (split 64)")

    # 2: the balanced schedule right after: its warp slots and arrival counters
    #    land on the stale partials of call 1
    b = H.make_case([900, 5, 257, 64, 1, 130], 8, 4, 64, "f16", seed=32)
    assert B.resolved_partition(6, 8, 4, 64, b.tables.shape[1], B.BALANCED) == B.BALANCED
    assert B.workspace_size(6, 8, 4, 64, b.tables.shape[1], B.BALANCED) > 0
    _check(b, B.BALANCED, "call 2 (balanced)")

    # 3: a batch of 256 sequences in a grid of 2048 CTAs: one pass, whose only
    #    scratch is the launch order written by the ordering kernel
    rng = np.random.default_rng(33)
    lens = np.clip(np.round(150 * np.exp(0.6 * rng.standard_normal(256))), 8, 1024).astype(np.int32)
    lens[[5, 77]] = [1024, 0]
    c = H.make_case(lens, 16, 8, 64, "bf16", seed=33)
    assert B.resolved_partition(256, 16, 8, 64, c.tables.shape[1]) == -1
    assert 0 < B.workspace_size(256, 16, 8, 64, c.tables.shape[1]) <= B.NOALLOC_SCRATCH_BYTES
    _check(c, 0, "call 3 (ordered one pass)")

    # 4: split again, another shape and fewer partitions (counters at a new offset)
    d = H.make_case([400, 17, 1200], 8, 8, 128, "f16", seed=34)
    _check(d, 256, "call 4 (split 256)")

    # 5: the shared-prefix schedule over parallel samples: its prefix plan,
    #    the partials of groups split into chunks and their counters all land
    #    on the stale contents of the calls before
    e, _ = H.sampling_case(6, 4, (70, 300), (0, 40), 8, 8, 128, "bf16", seed=35)
    assert B.resolved_partition(e.q.shape[0], 8, 8, 128, e.tables.shape[1], B.SHARED_PREFIX) == B.SHARED_PREFIX
    _check(e, B.SHARED_PREFIX, "call 5 (shared prefix)")
    assert B.device_status(clear=True) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    case = H.make_case([16], 8, 8, 128, "f16", seed=35)
    big_tables = torch.full((4096, 2048), -1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(4096, dtype=torch.int32, device="cuda")
    q = torch.zeros((4096, 8, 128), dtype=torch.float16, device="cuda")
    need = B.workspace_size(4096, 8, 8, 128, 2048, 16)
    assert need > B.NOALLOC_SCRATCH_BYTES
    out = torch.full_like(q, 7.0)
    torch.cuda.synchronize()
    with pytest.raises(B.PagedKVError) as exc:
        B.paged_attention_decode_noalloc(out, q, case.k_pool, case.v_pool, big_tables, lens, case.scale,
                                         partition_size=16)
    assert exc.value.status == 2 and "scratch" in str(exc.value)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0), "a rejected call launched work"
    assert B.device_status(clear=True) == 0
