"""Shared helpers of the GPU parity tests: seeded cases, oracle runs on host
copies of the inputs, and the attention tolerance.

Tolerance (fp16/bf16 I/O, fp32 accumulation, against the float64 oracle):
element-wise |got - want| <= 2e-3 + 1e-2 * |want|. A pure absolute 2e-3
bound cannot hold for bf16: one rounding of an output in [1, 2) to bf16 can
move it by up to 2^-8 = 3.9e-3. The combined bound keeps the absolute 2e-3
near zero (where a relative bound is meaningless) and allows the 1 %
relative error elsewhere; fp16 outputs additionally meet the plain 2e-3
absolute bound for |out| < 4.
"""

import numpy as np
import torch

import oracle.attention as OA
from paged_kv_cache_217_gb300 import workloads as W

ATOL = 2e-3
RTOL = 1e-2


def ensure_built():
    from paged_kv_cache_217_gb300 import build
    build.build()


def torch_dtype(dtype):
    return {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]


class DecodeCase:
    """Device tensors of one decode call plus what the oracle needs."""

    def __init__(self, q, k_pool, v_pool, tables, lens, scale, dtype):
        self.q, self.k_pool, self.v_pool = q, k_pool, v_pool
        self.tables, self.lens = tables, lens
        self.scale, self.dtype = scale, dtype

    @property
    def num_kv_heads(self):
        return self.k_pool.shape[1]

    def new_out(self):
        return torch.full_like(self.q, float("nan"))


def make_case(lens, hq, hkv, d, dtype, seed, device="cuda", pool_factor=1.2, extra_cols=0,
              scale=None):
    lens = np.asarray(lens, dtype=np.int32)
    nb = W.pool_size(lens, pool_factor) + 1
    tables, _ = W.scattered_tables(lens, nb, seed, extra_cols=extra_cols)
    k_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 7 + 1, device)
    v_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 7 + 2, device)
    q = W.normal_values((len(lens), hq, d), dtype, seed * 7 + 3, device)
    return DecodeCase(q, k_pool, v_pool, torch.from_numpy(tables).to(device),
                      torch.from_numpy(lens).to(device), scale if scale is not None else d ** -0.5, dtype)


def oracle_full(case):
    return OA.paged_attention_decode(
        W.to_numpy_storage(case.q, case.dtype), W.to_numpy_storage(case.k_pool, case.dtype),
        W.to_numpy_storage(case.v_pool, case.dtype), case.tables.cpu().numpy(), case.lens.cpu().numpy(),
        case.scale, case.num_kv_heads, case.dtype)


def oracle_sampled(case, pairs):
    """Oracle rows for a few (seq, q head) pairs without copying whole pools:
    each pair's KV head is sliced out and its used blocks gathered into a small
    sub-pool, with the table relabelled to match (relabelling physical ids does
    not change attention, which the oracle's own pins check)."""
    hq = case.q.shape[1]
    group = hq // case.num_kv_heads
    rows = {}
    lens = case.lens.cpu().numpy()
    tables = case.tables.cpu().numpy()
    for s, h in pairs:
        g = h // group
        L = int(lens[s])
        nb = -(-L // 16)
        ids = torch.from_numpy(tables[s, :nb].astype(np.int64)).to(case.k_pool.device)
        kp = case.k_pool[:, g].index_select(0, ids).unsqueeze(1)
        vp = case.v_pool[:, g].index_select(0, ids).unsqueeze(1)
        q = case.q[s, h].reshape(1, 1, -1)
        out = OA.paged_attention_decode(
            W.to_numpy_storage(q, case.dtype), W.to_numpy_storage(kp, case.dtype),
            W.to_numpy_storage(vp, case.dtype), np.arange(max(nb, 1), dtype=np.int32).reshape(1, -1),
            np.array([L], np.int32), case.scale, 1, case.dtype)
        rows[(s, h)] = out[0, 0]
    return rows


def errors(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    diff = np.abs(got - want)
    return {
        "max_abs": float(diff.max()) if diff.size else 0.0,
        "max_rel_floored": float((diff / np.maximum(np.abs(want), 1e-2)).max()) if diff.size else 0.0,
        "max_excess": float((diff - (ATOL + RTOL * np.abs(want))).max()) if diff.size else -1.0,
    }


def assert_attention_close(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    e = errors(got, want)
    assert e["max_excess"] <= 0.0, f"{what}: tolerance exceeded {e}"
    return e


def to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def sampling_case(num_prompts, n, prompt_range, tail_range, hq, hkv, d, dtype, seed):
    """Sequences from the block manager after parallel sampling (prompt added,
    forked n-1 times, tails appended with copy-on-write), pools filled with
    seeded values, copy-on-write pairs applied. Returns (case, trace)."""
    from paged_kv_cache_217_gb300 import binding as B
    trace = W.ParallelSamplingTrace("sampling", dtype, hq, hkv, d,
                                    np.random.default_rng(seed).integers(*prompt_range, size=num_prompts,
                                                                         endpoint=True).astype(np.int32),
                                    np.random.default_rng(seed + 1).integers(*tail_range, size=(num_prompts, n),
                                                                             endpoint=True).astype(np.int32))
    nb = trace.block_budget()
    bm = B.BlockManager(nb, W.shuffled_free_order(nb, seed))
    plan = W.drive_parallel_sampling(trace, bm)
    kp = W.normal_values((nb, hkv, 16, d), dtype, seed * 3 + 1, "cuda")
    vp = W.normal_values((nb, hkv, 16, d), dtype, seed * 3 + 2, "cuda")
    if plan.pairs:
        B.copy_blocks(kp, vp, torch.tensor(plan.pairs, dtype=torch.int64, device="cuda").reshape(-1, 2))
    mb = max(-(-L // 16) for L in plan.final_lens.values())
    tables, lens = bm.block_tables(plan.seq_ids, mb)
    q = W.normal_values((len(plan.seq_ids), hq, d), dtype, seed * 3 + 3, "cuda")
    return DecodeCase(q, kp, vp, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(), d ** -0.5,
                      dtype), trace
