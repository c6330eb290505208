"""The per-CTA tracing build (PKV_TRACE=1) and its timeline tool, run in a
separate process on a small and a full-size layer."""

import os
import re
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def trace_lib(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_217_gb300 import build
    out = str(tmp_path_factory.mktemp("trace_build"))
    return build.build(out_dir=out, defines=["PKV_TRACE=1"])


@pytest.mark.parametrize("workload,ctas", [("tiny", 16), ("llama3_8b", 2048)])
def test_timeline_of_one_decode(trace_lib, workload, ctas):
    res = subprocess.run([sys.executable, "-m", "paged_kv_cache_217_gb300.trace", "--lib", trace_lib,
                          "--workload", workload, "--calls", "3", "--replay"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = res.stdout.splitlines()
    # where the call's time goes: three positive intervals between the stamps
    anatomy = lines[0]
    assert "stamp -> first CTA" in anatomy, res.stdout
    parts = [float(x) for x in re.findall(r"(-?[0-9.]+) us", anatomy.split("stamp -> first CTA")[1])[:3]]
    assert len(parts) == 3, anatomy
    assert all(p > 0.0 for p in parts), anatomy
    assert f"{ctas} CTAs traced" in lines[1], res.stdout
    # every phase line is present and the mean lifetime is positive
    assert sum(1 for ln in lines if " us  median " in ln) == 6
    assert sum(1 for ln in lines if "modelled span" in ln) == 4, res.stdout
    life = [ln for ln in lines if ln.strip().startswith("lifetime")][0]
    assert float(life.split("mean")[1].split("us")[0]) > 0.0


def test_stamps_follow_the_stream():
    """pkv_trace_stamp writes the GPU clock when the stream reaches it: two
    stamps around a ~1 ms device sleep are at least 0.1 ms apart, in order."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_217_gb300 import binding as B
    words = torch.zeros(4, dtype=torch.int64, device="cuda")
    B.trace_stamp(words, 1)
    torch.cuda._sleep(2_000_000)
    B.trace_stamp(words, 3)
    torch.cuda.synchronize()
    w = words.cpu().tolist()
    assert w[0] == 0 and w[2] == 0
    assert w[3] - w[1] >= 100_000, w
    with pytest.raises(ValueError):
        B.trace_stamp(words.to(torch.int32), 0)
    with pytest.raises(ValueError):
        B.trace_stamp(words, 4)


def test_empty_grid_runs_in_stream_order():
    """pkv_trace_empty_grid launches a kernel of the given shape that does
    nothing: stamps around it are in order, the stream stays usable, and a
    decode-shaped grid (2048 CTAs x 96 threads, 50 KB of shared memory) and
    the largest shared-memory request both launch."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_217_gb300 import binding as B
    words = torch.zeros(2, dtype=torch.int64, device="cuda")
    B.trace_stamp(words, 0)
    B.trace_empty_grid("cuda", 2048, 96, 50224)
    B.trace_empty_grid("cuda", 152, 1024, 227 * 1024)
    B.trace_stamp(words, 1)
    torch.cuda.synchronize()
    w = words.cpu().tolist()
    assert 0 < w[0] <= w[1], w
    with pytest.raises(B.PagedKVError):
        B.trace_empty_grid("cuda", 1, 32, 227 * 1024 + 1)
    assert B.device_status(clear=True) == 0



def test_calibration_on_the_default_build():
    """--calibrate needs no trace build: it prints the decode call and the two
    empty launches (median and mean, both positive) and the stamp gap."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    res = subprocess.run([sys.executable, "-m", "paged_kv_cache_217_gb300.trace", "--calibrate",
                          "--workload", "tiny", "--calls", "20"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 4, res.stdout
    assert "decode call" in lines[0] and "1 CTA x 32 threads" in lines[1] and "16 CTAs x 96 threads" in lines[2]
    for ln in lines[:3]:
        med, mean = [float(x) for x in re.findall(r"([0-9.]+) us", ln)]
        assert med > 0.0 and mean > 0.0, ln
    assert float(re.findall(r"median ([0-9.]+) us", lines[3])[0]) > 0.0, lines[3]
