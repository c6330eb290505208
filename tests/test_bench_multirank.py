"""The multi-GPU bench path, on CPU: two gloo ranks combine their step times
with the same function bench.py uses under torchrun (max over ranks), and the
whole-job value counts every rank's bytes against the slowest rank's time.
The path has no exchange step (replicas), so this is all that N > 1 adds."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(times[rank])
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step():
    world = 2
    times = [[0.130, 0.160], [0.145, 0.150]]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
        got = dict(out)
    assert got[0] == got[1] == pytest.approx([0.145, 0.160])
    # every rank processed 909.5 MB; the job took the slowest rank's 0.145 ms
    assert bench.whole_job_gbs(909_475_840, got[0][0], world) == pytest.approx(2 * 909_475_840 / 0.145e-3 / 1e9)


def test_single_process_is_the_identity():
    assert bench.max_over_ranks([1.5, 2.0]) == [1.5, 2.0]


def test_reference_arm_on_a_non_zero_rank_does_no_work(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(bench, "build_workload", lambda *a, **k: pytest.fail("rank 1 must not build a workload"))
    bench.main(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"])
