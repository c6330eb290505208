"""Failure detection on the GPU without a GPU fault: a bounded wait that no
copy completes runs out, the device status word says so, and the context
keeps working. Bad indices are covered in test_gpu_decode / test_gpu_cache_ops."""

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


def test_wait_that_never_completes_times_out_and_is_reported():
    B.device_status(clear=True)
    B.selftest_bounded_wait(limit_us=2000)
    flags = B.device_status(clear=True)
    assert flags & 0x10, B.describe_device_flags(flags)
    # the context still works: a decode after the timeout matches the oracle
    case = H.make_case([40, 7], 4, 4, 64, "f16", seed=51)
    out = case.new_out()
    B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale)
    torch.cuda.synchronize()
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "after timeout")
    assert B.device_status(clear=True) == 0


def test_selftest_rejects_bad_limits():
    for bad in (0, 2_000_000):
        with pytest.raises(B.PagedKVError):
            B.selftest_bounded_wait(limit_us=bad)
