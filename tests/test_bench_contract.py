"""The benchmark's JSON line: the reference arm (the oracle on the host) on
CPU, and this library's arm on a GPU."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=900):
    res = subprocess.run([sys.executable, "bench.py"] + args, cwd=ROOT, capture_output=True, text=True,
                         timeout=timeout)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3",
              "--reference-budget", "2"])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and 1 <= d["cpu_baseline"]["cores"] <= os.cpu_count()
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_our_arm_line():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _run(["--workload", "llama3_8b", "--steps", "20", "--warmup", "3", "--no-cpu-baseline"])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert "workload" in d["config"] and d["dtype"] == "bf16"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    e = d["e2e"]
    assert e["unit"] == "GB/s" and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # cache write + ranking kernel (256 sequences) + decode per step
    assert d["gpu_launches"] == 20 * 3
    pc = d["per_config"]["configs"]
    assert sorted(pc) == ["llama13b", "llama3_8b", "opt175b_long", "opt66b_sampling"]
    for name, e in pc.items():
        assert e["decode_us"] > 0 and abs(e["frac"] - e["achieved"] / d["per_config"]["peak"]) < 1e-3, name
    # the sampling batch shares prompt blocks: its roofline counts them once
    assert pc["opt66b_sampling"]["algorithmic_bytes_per_launch"] < pc["opt66b_sampling"]["logical_bytes_per_launch"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_oracle_shares_cover_every_sequence_and_head_once():
    import numpy as np
    import bench
    for hkv, seqs, cores in [(96, 1, 16), (8, 256, 16), (8, 3, 16), (4, 4, 1), (40, 64, 72), (8, 1, 5)]:
        lens = np.arange(1, seqs + 1, dtype=np.int32) * 7
        shares = bench._shares({"seqs": seqs, "lens": lens}, hkv, cores)
        seen = np.zeros((seqs, hkv), int)
        for h0, h1, s0, s1 in shares:
            seen[s0:s1, h0:h1] += 1
        assert (seen == 1).all(), (hkv, seqs, cores)
        assert len(shares) <= max(cores, 1)
