"""The decode entry point that allocates nothing, checked against the regular one.

pkv_paged_attention_decode_noalloc serves callers that cannot allocate device
memory while they decode (an engine whose allocator already holds nearly all
HBM for the KV pool, or host code that must not call cudaMalloc/cudaFree and
risk a device synchronisation). Its split-K scratch is a fixed array inside
the library. These tests call it through the C ABI twice in a row, on
different inputs, and compare each result with the workspace-taking entry
point within the attention tolerance of the other GPU tests.

This file is collected last on purpose: a run that stops at the first failure
has already run every other test when it gets here.
"""

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
    yield


def _both(case, partition):
    ref = case.new_out()
    B.paged_attention_decode(ref, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             partition_size=partition)
    got = case.new_out()
    B.paged_attention_decode_noalloc(got, case.q, case.k_pool, case.v_pool, case.tables, case.lens,
                                     case.scale, partition_size=partition)
    torch.cuda.synchronize()
    return H.to_f64(got), H.to_f64(ref)


def test_noalloc_matches_the_workspace_entry_on_two_calls_in_a_row():
    # first call: long, split contexts (GQA, bf16) fill a large part of the scratch
    a = H.make_case([2048, 700, 33, 1, 0, 1500, 517, 16], 32, 8, 128, "bf16", seed=31)
    need_a = B.workspace_size(8, 32, 8, 128, a.tables.shape[1], 64)
    assert 0 < need_a <= B.NOALLOC_SCRATCH_BYTES
    got, ref = _both(a, 64)
    H.assert_attention_close(got, ref, "no-alloc call 1")
    # second call: different shapes and fewer partitions; stale scratch contents
    # from the first call must not leak into the result
    b = H.make_case([900, 5, 257, 64], 8, 8, 64, "f16", seed=32)
    got, ref = _both(b, 0)
    H.assert_attention_close(got, ref, "no-alloc call 2")
    assert B.device_status(clear=True) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    case = H.make_case([16], 8, 8, 128, "f16", seed=33)
    big_tables = torch.full((4096, 2048), -1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(4096, dtype=torch.int32, device="cuda")
    q = torch.zeros((4096, 8, 128), dtype=torch.float16, device="cuda")
    need = B.workspace_size(4096, 8, 8, 128, 2048, 16)
    assert need > B.NOALLOC_SCRATCH_BYTES
    with pytest.raises(B.PagedKVError) as exc:
        B.paged_attention_decode_noalloc(torch.empty_like(q), q, case.k_pool, case.v_pool, big_tables, lens,
                                         case.scale, partition_size=16)
    assert exc.value.status == 2 and "scratch" in str(exc.value)
