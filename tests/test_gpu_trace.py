"""The per-CTA tracing build (PKV_TRACE=1) and its timeline tool, run in a
separate process on a small and a full-size layer."""

import os
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
                          "--workload", workload, "--calls", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = res.stdout.splitlines()
    assert f"{ctas} CTAs traced" in lines[0], res.stdout
    # every phase line is present and the mean lifetime is positive
    assert sum(1 for ln in lines if " us  median " in ln) == 6
    life = [ln for ln in lines if ln.strip().startswith("lifetime")][0]
    assert float(life.split("mean")[1].split("us")[0]) > 0.0
