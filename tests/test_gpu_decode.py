"""GPU parity of paged_attention_decode (through the C ABI) against the fp64 oracle.

Small cases compare every output element; the full-size workloads compare
sampled (sequence, head) outputs, in the launch configuration the benchmark
times (automatic partition choice)."""

import numpy as np
import pytest
import torch

import helpers as H
import oracle.attention as OA
from oracle.block_manager import OracleBlockManager
import oracle.cache_ops as OC
from paged_kv_cache_217_gb300 import binding as B
from paged_kv_cache_217_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    H.ensure_built()
    B.device_status(clear=True)
    yield
    flags = B.device_status(clear=True)
    assert flags == 0, f"device flags raised: {B.describe_device_flags(flags)}"


def _run(case, partition=0):
    out = case.new_out()
    B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             partition_size=partition)
    torch.cuda.synchronize()
    return out


# ---------------------------------------------------------------------------
# tiny decode (batch 4, L = 5, 17, 33, 64, 4 heads, d 64, fp16), tables from
# the block manager over a seeded permutation of a 64-block pool, then one
# new token per sequence written with reshape_and_cache
# ---------------------------------------------------------------------------
def test_tiny_decode_with_reshape():
    shape = W.tiny_decode()
    order = W.shuffled_free_order(64, 0)
    bm, obm = B.BlockManager(64, order), OracleBlockManager(64, initial_free_order=order)
    for s, L in enumerate(shape.context_lens.tolist()):
        bm.add_seq(s, L)
        obm.add_seq(s, L)
    tables, lens = bm.block_tables(range(4), 5)
    dev = "cuda"
    kp = W.normal_values((64, 4, 16, 64), "f16", 1, dev)
    vp = W.normal_values((64, 4, 16, 64), "f16", 2, dev)
    q = W.normal_values((4, 4, 64), "f16", 3, dev)
    case = H.DecodeCase(q, kp, vp, torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev),
                        1.0 / 8.0, "f16")
    want = H.oracle_full(case)
    for part in (0, -1, 16, 32):
        e = H.assert_attention_close(H.to_f64(_run(case, part)), want, f"tiny part={part}")
        assert e["max_abs"] <= 2e-3  # fp16 outputs meet the plain absolute bound

    # one new token per sequence into its next slot (L=64 needs a fifth block)
    slots, pairs = bm.append_slots(range(4))
    assert slots.tolist() == [obm.append_slot(s)[0] for s in range(4)] and pairs.size == 0
    knew = W.normal_values((4, 4, 64), "f16", 4, dev)
    vnew = W.normal_values((4, 4, 64), "f16", 5, dev)
    k_before, v_before = W.to_numpy_storage(kp, "f16"), W.to_numpy_storage(vp, "f16")
    B.reshape_and_cache(knew, vnew, kp, vp, torch.from_numpy(slots).to(dev))
    torch.cuda.synchronize()
    ok, ov = OC.reshape_and_cache(W.to_numpy_storage(knew, "f16"), W.to_numpy_storage(vnew, "f16"),
                                  k_before, v_before, slots)
    assert np.array_equal(W.to_numpy_storage(kp, "f16").view(np.uint16), ok.view(np.uint16))
    assert np.array_equal(W.to_numpy_storage(vp, "f16").view(np.uint16), ov.view(np.uint16))
    tables2, lens2 = bm.block_tables(range(4), 5)
    assert lens2.tolist() == [6, 18, 34, 65]
    case2 = H.DecodeCase(q, kp, vp, torch.from_numpy(tables2).to(dev), torch.from_numpy(lens2).to(dev),
                         1.0 / 8.0, "f16")
    H.assert_attention_close(H.to_f64(_run(case2)), H.oracle_full(case2), "tiny after reshape")


# ---------------------------------------------------------------------------
# shapes, dtypes, group sizes and partitions, every element compared
# ---------------------------------------------------------------------------
RAGGED = [1, 15, 16, 17, 31, 33, 100, 0, 255, 257, 700]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (32, 8), (6, 2), (16, 2), (3, 1)])
def test_decode_matches_oracle(dtype, d, hq, hkv):
    case = H.make_case(RAGGED, hq, hkv, d, dtype, seed=d + hq + hkv, extra_cols=3)
    want = H.oracle_full(case)
    for part in (0, -1, -2, 64, 512):
        H.assert_attention_close(H.to_f64(_run(case, part)), want, f"{dtype} d={d} {hq}/{hkv} part={part}")


def test_zero_length_rows_are_zero_and_others_untouched():
    case = H.make_case([0, 5, 0, 40], 8, 4, 128, "bf16", seed=3)
    out = _run(case)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "zero rows")


def test_scores_large_and_scale_extremes():
    # large logits: values x 8 make exp() span many orders of magnitude
    case = H.make_case([300, 47, 1000], 8, 8, 128, "f16", seed=4, scale=1.0)
    case.q.mul_(4)
    case.k_pool.mul_(2)
    H.assert_attention_close(H.to_f64(_run(case)), H.oracle_full(case), "large logits")
    H.assert_attention_close(H.to_f64(_run(case, 16)), H.oracle_full(case), "large logits split 16")


def test_split_calls_with_different_shapes_share_one_workspace():
    # The binding reuses one workspace; a later call's partition counters may sit
    # where an earlier call left partials, so every split call must start clean.
    small = H.make_case([700, 40], 8, 2, 128, "bf16", seed=41)
    large = H.make_case([600 + 37 * i for i in range(40)], 8, 8, 128, "bf16", seed=42)
    want_small, want_large = H.oracle_full(small), H.oracle_full(large)
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    for case, want in ((small, want_small), (large, want_large), (small, want_small), (large, want_large)):
        out = case.new_out()
        B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                                 partition_size=32, workspace=ws)
        torch.cuda.synchronize()
        H.assert_attention_close(H.to_f64(out), want, "shared workspace")
        ws[: 32 << 20].fill_(0x7f)   # stale garbage everywhere the next call may look


@pytest.mark.parametrize("lens,hq,hkv,d,dtype", [
    ([30000], 4, 1, 128, "bf16"),                        # one item spread over hundreds of warps
    ([3] * 500 + [1, 16, 17, 0], 8, 8, 64, "f16"),       # hundreds of tiny items
    ([900, 901, 17], 32, 8, 128, "f16"),                 # GQA, few long items
    ([5, 0, 0, 33], 16, 2, 256, "bf16"),                 # group 8, head_dim 256, empty sequences
])
def test_balanced_schedule_matches_oracle(lens, hq, hkv, d, dtype):
    case = H.make_case(lens, hq, hkv, d, dtype, seed=len(lens) + d)
    assert B.resolved_partition(len(lens), hq, hkv, d, case.tables.shape[1], -2) == B.BALANCED
    want = H.oracle_full(case)
    H.assert_attention_close(H.to_f64(_run(case, -2)), want, f"balanced {lens[:3]}")
    H.assert_attention_close(H.to_f64(_run(case)), want, f"auto {lens[:3]}")


@pytest.mark.parametrize("S", [2048, 2049])
def test_batch_size_limit_of_the_balanced_schedule(S):
    # The balanced schedule keeps its prefix sums in shared memory: 2048 sequences
    # fit, 2049 are refused (nothing launched); the automatic choice runs both.
    rng = np.random.default_rng(S)
    lens = rng.integers(0, 300, size=S).astype(np.int32)
    case = H.make_case(lens, 8, 2, 128, "bf16", seed=S)
    if S <= 2048:
        out = _run(case, -2)
        _check_sampled(case, out, 24, seed=S)
    else:
        with pytest.raises(B.PagedKVError) as exc:
            _run(case, -2)
        assert exc.value.status == 2
    out = _run(case)
    _check_sampled(case, out, 24, seed=S + 1)
    zero = np.flatnonzero(lens == 0)
    if zero.size:
        assert torch.all(out[torch.from_numpy(zero).cuda()] == 0)


# ---------------------------------------------------------------------------
# invariants the pages fix
# ---------------------------------------------------------------------------
def test_physical_permutation_is_bit_identical():
    case = H.make_case([37, 300, 1000, 12], 32, 8, 128, "bf16", seed=5, pool_factor=2.0)
    base = _run(case)
    nb = case.k_pool.shape[0]
    pi = torch.from_numpy(np.random.default_rng(9).permutation(nb)).to("cuda")
    kp2 = torch.empty_like(case.k_pool)
    vp2 = torch.empty_like(case.v_pool)
    kp2[pi] = case.k_pool
    vp2[pi] = case.v_pool
    t2 = torch.where(case.tables >= 0, pi[case.tables.clamp(min=0).long()].int(), case.tables)
    moved = H.DecodeCase(case.q, kp2, vp2, t2.contiguous(), case.lens, case.scale, case.dtype)
    assert torch.equal(_run(moved), base)


def test_partition_size_invariance():
    case = H.make_case([5000, 4097, 513, 64], 8, 8, 128, "f16", seed=6)
    outs = [H.to_f64(_run(case, p)) for p in (-1, 16, 512, 1024, 0)]
    want = H.oracle_full(case)
    for o in outs:
        H.assert_attention_close(o, want, "partition")
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 4e-3


def test_long_partitions_on_few_ctas():
    """Grids of at most 1024 CTAs run 6-warp rings when each CTA streams a
    long stretch: one pass, and split grids whose partitions hold at least
    12288 tokens (12288 and 16384 here); 512-token partitions and the
    library's own choice keep 4 warps. All against the oracle."""
    case = H.make_case([25000, 12289], 2, 2, 128, "bf16", seed=21)
    want = H.oracle_full(case)
    outs = {p: H.to_f64(_run(case, p)) for p in (-1, 12288, 16384, 512, 0)}
    for p, o in outs.items():
        H.assert_attention_close(o, want, f"partition {p}")


def test_cow_siblings_bit_identical_over_shared_prefix():
    hkv, d, prompt, n = 8, 128, 517, 4
    nb = 200
    order = W.shuffled_free_order(nb, 1)
    bm = B.BlockManager(nb, order)
    bm.add_seq(0, prompt)
    for c in range(1, n):
        bm.fork(0, c)
    kp = W.normal_values((nb, hkv, 16, d), "f16", 11, "cuda")
    vp = W.normal_values((nb, hkv, 16, d), "f16", 12, "cuda")
    slots, pairs = bm.append_slots(range(n))
    assert pairs.shape == (n - 1, 2)
    k_before = W.to_numpy_storage(kp, "f16")
    B.copy_blocks(kp, vp, torch.from_numpy(pairs).to("cuda"))
    knew = W.normal_values((n, hkv, d), "f16", 13, "cuda")
    B.reshape_and_cache(knew, knew, kp, vp, torch.from_numpy(slots).to("cuda"))
    torch.cuda.synchronize()
    k_after = W.to_numpy_storage(kp, "f16")
    for src, dst in pairs.tolist():
        assert np.array_equal(k_after[dst, :, :prompt % 16], k_before[src, :, :prompt % 16])
    tables, lens = bm.block_tables(range(n), 40)
    q = W.normal_values((1, hkv, d), "f16", 14, "cuda").expand(n, hkv, d).contiguous()
    shared = H.DecodeCase(q, kp, vp, torch.from_numpy(tables).cuda(),
                          torch.full((n,), prompt, dtype=torch.int32, device="cuda"), d ** -0.5, "f16")
    for partition in (0, B.SHARED_PREFIX):   # the default schedule and the shared-prefix one
        out = _run(shared, partition)
        for s in range(1, n):
            assert torch.equal(out[s], out[0]), f"partition {partition}: sibling {s}"
    grown = H.DecodeCase(q, kp, vp, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                         d ** -0.5, "f16")
    H.assert_attention_close(H.to_f64(_run(grown)), H.oracle_full(grown), "siblings after append")


# ---------------------------------------------------------------------------
# device-side index checks: flagged, never faulting
# ---------------------------------------------------------------------------
def test_bad_device_indices_are_flagged():
    case = H.make_case([40, 20], 4, 4, 64, "f16", seed=7)
    B.device_status(clear=True)
    bad = case.tables.clone()
    bad[0, 1] = case.k_pool.shape[0] + 5        # outside the pool
    B.paged_attention_decode(case.new_out(), case.q, case.k_pool, case.v_pool, bad, case.lens, case.scale)
    assert B.device_status(clear=True) & 0x1
    lens = case.lens.clone()
    lens[1] = 10_000                              # longer than the table allows
    B.paged_attention_decode(case.new_out(), case.q, case.k_pool, case.v_pool, case.tables, lens, case.scale)
    assert B.device_status(clear=True) & 0x2
    out = _run(case)                              # a clean call raises nothing
    assert B.device_status(clear=True) == 0
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "after flags")


# ---------------------------------------------------------------------------
# full-size workloads, sampled outputs, automatic partitioning (bench config)
# ---------------------------------------------------------------------------
def _sample_pairs(rng, S, hq, k, lens=None):
    """(sequence, query head) pairs to check: one random head of every
    sequence, the first and last head of the longest sequence (and of the
    first and last sequence), plus random pairs up to k in all."""
    pairs = {(0, 0), (S - 1, hq - 1)}
    for s in range(S):
        pairs.add((s, int(rng.integers(hq))))
    if lens is not None and S > 0:
        longest = int(np.argmax(lens))
        pairs |= {(longest, 0), (longest, hq - 1)}
    while len(pairs) < k:
        pairs.add((int(rng.integers(S)), int(rng.integers(hq))))
    return sorted(pairs)


def _check_sampled(case, out, k, seed):
    rng = np.random.default_rng(seed)
    lens = case.lens.cpu().numpy()
    pairs = _sample_pairs(rng, case.q.shape[0], case.q.shape[1], k, lens)
    assert {s for s, _ in pairs} == set(range(case.q.shape[0]))
    want = H.oracle_sampled(case, pairs)
    got = H.to_f64(out)
    for (s, h), w in want.items():
        H.assert_attention_close(got[s, h], w, f"seq {s} head {h}")
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("name", ["llama13b", "llama3_8b", "opt175b_long"])
def test_full_size_decode_sampled(name):
    shape = W.CONFIGS[name](0)
    case = H.make_case(shape.context_lens, shape.num_q_heads, shape.num_kv_heads, shape.head_dim,
                       shape.dtype, seed=0)
    out = _run(case)
    _check_sampled(case, out, 24 if name == "opt175b_long" else 40, seed=1)
    del case, out
    torch.cuda.empty_cache()


def test_full_size_long_context_split_512():
    # the long-context layer with its own stated schedule: split-K partitions of
    # 512 tokens (up to 64 per sequence) merged by log-sum-exp in the kernel
    shape = W.CONFIGS["opt175b_long"](0)
    case = H.make_case(shape.context_lens, shape.num_q_heads, shape.num_kv_heads, shape.head_dim,
                       shape.dtype, seed=0)
    assert B.resolved_partition(8, 96, 96, 128, case.tables.shape[1], 512) == 512
    out = _run(case, 512)
    _check_sampled(case, out, 24, seed=3)
    # the split result agrees with the one-pass result to fp32 rounding
    one = _run(case, -1)
    H.assert_attention_close(H.to_f64(out), H.to_f64(one), "split 512 against one pass")
    del case, out, one
    torch.cuda.empty_cache()


def test_full_size_parallel_sampling():
    trace = W.opt66b_parallel_sampling(0)
    nb = trace.block_budget()
    bm = B.BlockManager(nb, W.shuffled_free_order(nb, 0))
    plan = W.drive_parallel_sampling(trace, bm)
    dev = "cuda"
    kp = W.normal_values((nb, 72, 16, 128), "f16", 21, dev)
    vp = W.normal_values((nb, 72, 16, 128), "f16", 22, dev)
    k_host_blocks = {}
    for src, dst in plan.pairs:
        k_host_blocks[src] = kp[src].clone()
    B.check_copy_pairs(plan.pairs, nb)
    B.copy_blocks(kp, vp, torch.tensor(plan.pairs, dtype=torch.int64, device=dev).reshape(-1, 2))
    for src, dst in plan.pairs:
        assert torch.equal(kp[dst], k_host_blocks[src])
    all_slots = np.concatenate([sl for _, sl in plan.step_slots]) if plan.step_slots else np.zeros(0, np.int64)
    knew = W.normal_values((all_slots.size, 72, 128), "f16", 23, dev)
    vnew = W.normal_values((all_slots.size, 72, 128), "f16", 24, dev)
    B.reshape_and_cache(knew, vnew, kp, vp, torch.from_numpy(all_slots).to(dev))
    tables, lens = bm.block_tables(plan.seq_ids, max(-(-L // 16) for L in plan.final_lens.values()))
    assert lens.tolist() == [plan.final_lens[s] for s in plan.seq_ids]
    q = W.normal_values((len(plan.seq_ids), 72, 128), "f16", 25, dev)
    case = H.DecodeCase(q, kp, vp, torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev),
                        128 ** -0.5, "f16")
    out = _run(case)
    _check_sampled(case, out, 24, seed=2)
    # a sibling's shared prompt blocks are the very same physical blocks
    n = trace.n
    t = tables
    for i in range(trace.prompt_lens.shape[0]):
        full = int(trace.prompt_lens[i]) // 16
        for c in range(1, n):
            assert np.array_equal(t[i * n + c, :full], t[i * n, :full])


@pytest.mark.parametrize("dtype,d", [("f16", 64), ("bf16", 128)])
@pytest.mark.parametrize("partition", [0, 32])
def test_wide_grid_ring_shape(dtype, d, partition):
    # 256 sequences x 40 KV heads = 10240 CTAs: the CUDA-core kernel runs its
    # six-warp, one-stage ring (with 32-token partitions the split grid is wider still)
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 120, 256).astype(np.int32)
    case = H.make_case(lens, 40, 40, d, dtype, seed=31)
    out = _run(case, partition)
    _check_sampled(case, out, 40, seed=6)
    assert B.device_status(clear=True) == 0


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("bf16", 256)])
@pytest.mark.parametrize("partition", [0, 16, 48])
def test_every_partial_tile_size_on_the_tensor_cores(dtype, d, partition):
    # lengths 1..48: the last tile of a sequence (or of a split part) holds
    # every count of valid rows from 1 to 16, copied as boxes of 16, 8 and 4 rows
    lens = np.arange(1, 49, dtype=np.int32)
    case = H.make_case(lens, 8, 2, d, dtype, seed=60 + d)
    out = _run(case, partition)
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), f"partial tiles d={d} p={partition}")
    assert B.device_status(clear=True) == 0


PLAN_MAGIC = 0x504b5631  # the first word of a launch plan's header


def _dispatch_order(lens, max_len, short_last=True):
    """The row order the ordering kernel promises, restated on the host: tiles
    t = ceil(min(max(L, 0), max_len) / 16), mean over the batch; sequences with
    t >= 2 x mean first, then (with short_last) those above 5/8 of the mean,
    then the rest, each in natural order."""
    t = [(min(max(int(L), 0), max_len) + 15) // 16 for L in lens]
    S, total = len(t), sum(t)
    longs = [s for s in range(S) if 2 * t[s] * S >= 4 * total]
    shorts = [s for s in range(S) if short_last and s not in set(longs) and 8 * t[s] * S <= 5 * total]
    rest = [s for s in range(S) if s not in set(longs) and s not in set(shorts)]
    return longs + rest + shorts


def _plan_at(need, S):
    """Offset of the plan's order array: the plan region ends the workspace with
    a 16-byte header, int32[S] (16-byte rounded), then int4[2 S] of rows."""
    return need - 32 * S - (4 * S + 15) // 16 * 16


def _plan_rows_want(order, lens, tables):
    """The rows the plan promises, rank by rank: {sequence, its length, its
    first six block ids (-1 past the table's width)}."""
    t = tables.cpu().numpy()
    rows = []
    for s in order:
        ids = [int(t[s, i]) if i < t.shape[1] else -1 for i in range(6)]
        rows.append([s, int(lens[s])] + ids)
    return rows


@pytest.mark.parametrize("S,hkv,seed", [(128, 8, 0), (150, 4, 1), (256, 8, 2), (1024, 4, 3)])
def test_ordering_kernel_writes_the_promised_order(S, hkv, seed):
    # the order array (int32[S] after a 16-byte header) and the rows behind
    # it (int4[2 S], the last bytes of the workspace, after any split-K
    # scratch) are index work: they must equal the host restatement exactly
    rng = np.random.default_rng(40 + seed)
    lens = np.clip(np.round(150 * np.exp(0.6 * rng.standard_normal(S))), 8, 1024).astype(np.int32)
    lens[rng.integers(0, S, 3)] = 0
    lens[rng.integers(0, S, 2)] = 1024
    case = H.make_case(lens, 2 * hkv, hkv, 64, "f16", seed=50 + seed)
    mb = case.tables.shape[1]
    need = B.workspace_size(S, 2 * hkv, hkv, 64, mb)
    at = _plan_at(need, S)
    assert at >= 16 and at % 16 == 0
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(case.q)
    B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             workspace=ws)
    torch.cuda.synchronize()
    got = ws[at:at + 4 * S].view(torch.int32).cpu().tolist()
    want = _dispatch_order(lens.tolist(), mb * 16)
    assert got == want
    assert ws[at - 16:at].view(torch.int32).cpu().tolist() == [PLAN_MAGIC, S, 0, 0]
    assert sorted(got) == list(range(S))
    rows = ws[need - 32 * S:need].view(torch.int32).view(S, 8).cpu().tolist()
    assert rows == _plan_rows_want(want, lens, case.tables)
    _check_sampled(case, out, 16, seed=seed)
    assert B.device_status(clear=True) == 0


@pytest.mark.parametrize("dtype,hq,hkv,d", [("f16", 8, 4, 64), ("bf16", 4, 4, 128)])
def test_batch_ranked_once_for_the_grid(dtype, hq, hkv, d):
    # 150 sequences (128..1024) in a grid of at most 4096 CTAs: the long-first
    # order comes from the one-CTA ordering kernel; a few long sequences among
    # short ones make the order differ from the natural one
    rng = np.random.default_rng(8)
    lens = rng.integers(1, 60, 150).astype(np.int32)
    lens[[7, 90, 149]] = [900, 700, 1200]
    lens[20] = 0
    case = H.make_case(lens, hq, hkv, d, dtype, seed=17)
    assert B.workspace_size(150, hq, hkv, d, case.tables.shape[1]) > 0
    out = _run(case)
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "ordered batch")
    assert B.device_status(clear=True) == 0


# ---------------------------------------------------------------------------
# launch plans: made once per decode step, used by every layer's decode
# ---------------------------------------------------------------------------
def _lognormal_lens(S, seed, median=150, sigma=0.6, hi=1024):
    rng = np.random.default_rng(seed)
    lens = np.clip(np.round(median * np.exp(sigma * rng.standard_normal(S))), 1, hi).astype(np.int32)
    lens[rng.integers(0, S, 2)] = hi
    lens[rng.integers(0, S, 2)] = 0
    return lens


@pytest.mark.parametrize("S,hq,hkv,d,dtype,part", [(64, 40, 40, 128, "bf16", 0), (256, 32, 8, 128, "bf16", 0),
                                                   (150, 8, 4, 64, "f16", 0), (40, 16, 8, 128, "f16", 0),
                                                   (320, 16, 2, 256, "bf16", 0), (180, 8, 4, 64, "bf16", 0),
                                                   (200, 4, 4, 64, "bf16", 256), (300, 4, 4, 64, "bf16", 128)])
def test_planned_decode_matches_the_oracle_and_the_unplanned_call(S, hq, hkv, d, dtype, part):
    lens = _lognormal_lens(S, seed=S + d)
    case = H.make_case(lens, hq, hkv, d, dtype, seed=S + hq)
    mb = case.tables.shape[1]
    need = B.workspace_size(S, hq, hkv, d, mb, part)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    B.paged_attention_plan(case.lens, case.tables, hq, hkv, d, part, workspace=ws)
    parts = 1 if part == 0 else -(-mb * 16 // part)
    if S * hkv * parts <= 4096:     # a grid that starts long sequences first has a plan
        at = _plan_at(need, S)
        assert ws[at - 16:at].view(torch.int32).cpu().tolist() == [PLAN_MAGIC, S, 0, 0]
        # smaller batches keep two buckets, batches of 128+ put the shortest last
        order = ws[at:at + 4 * S].view(torch.int32).cpu().tolist()
        assert order == _dispatch_order(lens.tolist(), mb * 16, S >= 128)
    outs = []
    for layer in range(2):          # two layers of one step share the plan
        out = case.new_out()
        B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                                 partition_size=part, workspace=ws, planned=True)
        outs.append(out)
    plain = _run(case, part)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], plain)
    H.assert_attention_close(H.to_f64(outs[0]), H.oracle_full(case), f"planned S={S}")
    assert B.device_status(clear=True) == 0


def test_planned_decode_without_a_plan_is_flagged_and_still_correct():
    lens = _lognormal_lens(200, seed=5)
    case = H.make_case(lens, 16, 8, 128, "bf16", seed=77)
    mb = case.tables.shape[1]
    ws = torch.full((B.workspace_size(200, 16, 8, 128, mb),), 0x5A, dtype=torch.uint8, device="cuda")
    out = case.new_out()
    B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             workspace=ws, planned=True)
    torch.cuda.synchronize()
    assert B.device_status(clear=True) == 0x20          # BAD_PLAN: natural order instead
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "no plan")


def test_a_plan_of_other_lengths_is_still_correct():
    lens = _lognormal_lens(256, seed=6)
    case = H.make_case(lens, 32, 8, 128, "bf16", seed=78)
    mb = case.tables.shape[1]
    ws = torch.empty((B.workspace_size(256, 32, 8, 128, mb),), dtype=torch.uint8, device="cuda")
    other = torch.from_numpy(np.roll(lens, 17)).cuda()   # same batch size, other lengths
    B.paged_attention_plan(other, case.tables, 32, 8, 128, workspace=ws)
    out = case.new_out()
    B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             workspace=ws, planned=True)
    torch.cuda.synchronize()
    assert B.device_status(clear=True) == 0
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "stale plan")


@pytest.mark.parametrize("change", ["all ids", "one id", "lengths and ids"])
def test_a_plan_of_other_tables_is_still_correct(change):
    """The tensor-core kernel starts its first copies from the plan's rows and
    checks them against the sequence's own length and ids: a plan made from
    other tables (every id, a single id of the first six, or lengths and
    ids) gives the same outputs as a fresh plan, bit for bit, and no flag."""
    lens = _lognormal_lens(256, seed=9)
    case = H.make_case(lens, 32, 8, 128, "bf16", seed=79)
    mb = case.tables.shape[1]
    need = B.workspace_size(256, 32, 8, 128, mb)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    B.paged_attention_plan(case.lens, case.tables, 32, 8, 128, workspace=ws)
    fresh = case.new_out()
    B.paged_attention_decode(fresh, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             workspace=ws, planned=True)
    tables = case.tables.clone()
    plan_lens = case.lens
    nb = case.k_pool.shape[0]
    if change == "all ids":
        tables = torch.where(tables >= 0, (tables + 7) % nb, tables)
    elif change == "one id":
        long_rows = (case.lens > 16 * 5).nonzero().flatten()
        tables[long_rows, 5] = (tables[long_rows, 5] + 1) % nb
    else:
        tables = torch.roll(tables, 3, dims=0)
        plan_lens = torch.roll(case.lens, 3)
    B.paged_attention_plan(plan_lens, tables, 32, 8, 128, workspace=ws)
    stale = case.new_out()
    B.paged_attention_decode(stale, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             workspace=ws, planned=True)
    torch.cuda.synchronize()
    assert B.device_status(clear=True) == 0
    assert torch.equal(stale, fresh)
    H.assert_attention_close(H.to_f64(stale), H.oracle_full(case), f"plan of other tables ({change})")


@pytest.mark.parametrize("mb", [1, 3, 5])
def test_plan_rows_of_narrow_tables(mb):
    """Tables narrower than the six block ids of a plan row: the row holds -1
    past the table, the speculative start stops there and the rest of the
    first tiles come from the sequence's own ids; one pass (-1) on the
    tensor cores, exact against the oracle and against the unplanned call."""
    rng = np.random.default_rng(30 + mb)
    S = 200
    lens = rng.integers(0, 16 * mb + 1, S).astype(np.int32)
    case = H.make_case(lens, 8, 2, 64, "bf16", seed=90 + mb)
    assert case.tables.shape[1] == mb
    need = B.workspace_size(S, 8, 2, 64, mb, -1)
    ws = torch.full((need,), 0x3C, dtype=torch.uint8, device="cuda")
    B.paged_attention_plan(case.lens, case.tables, 8, 2, 64, -1, workspace=ws)
    torch.cuda.synchronize()
    order = ws[_plan_at(need, S):_plan_at(need, S) + 4 * S].view(torch.int32).cpu().tolist()
    rows = ws[need - 32 * S:need].view(torch.int32).view(S, 8).cpu().tolist()
    assert rows == _plan_rows_want(order, lens, case.tables)
    out = case.new_out()
    B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             partition_size=-1, workspace=ws, planned=True)
    torch.cuda.synchronize()
    assert B.device_status(clear=True) == 0
    assert torch.equal(out, _run(case, -1))
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), f"narrow tables ({mb} blocks)")


def test_a_plan_without_tables_names_no_sequence():
    """pkv_paged_attention_plan with NULL block_tables (allowed outside the
    shared-prefix schedule) writes rows that name no sequence; the decode
    reads every length and id itself, with the same outputs."""
    lens = _lognormal_lens(200, seed=10)
    case = H.make_case(lens, 16, 4, 128, "f16", seed=80)
    S, mb = case.tables.shape
    need = B.workspace_size(S, 16, 4, 128, mb)
    ws = torch.full((need,), 0x11, dtype=torch.uint8, device="cuda")
    st = B.lib().pkv_paged_attention_plan(case.lens.data_ptr(), None, S, 16, 4, 128, mb, 0, ws.data_ptr(), need,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    rows = ws[need - 32 * S:need].view(torch.int32).view(S, 8).cpu().numpy()
    assert (rows[:, 0] == -1).all() and (rows[:, 2:] == -1).all()
    out = case.new_out()
    B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             workspace=ws, planned=True)
    torch.cuda.synchronize()
    assert B.device_status(clear=True) == 0
    assert torch.equal(out, _run(case))
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "plan without tables")


# ---------------------------------------------------------------------------
# the shared-prefix schedule: sibling sequences read their shared prompt
# blocks once per group
# ---------------------------------------------------------------------------
PREFIX_MAGIC = 0x504B5831  # the first word of a prefix plan's header


_sampling_case = H.sampling_case


def _prefix_layout(S, hq, hkv, d):
    # partials of up to 4 chunks a group (fp32 acc[d], (max, sum)) and one
    # counter per (sequence, KV head), then the prefix plan: header int4,
    # groups int4[S / 2], chunks int4[S], the other sequences int32[S]
    split = (S * hq * 4 * (4 * d + 8) + 4 * S * hkv + 15) // 16 * 16
    groups = split + 16
    chunks = groups + max(S // 2, 1) * 16
    others = chunks + 16 * S
    return dict(header=split, groups=groups, chunks=chunks, others=others, total=others + (4 * S + 15) // 16 * 16)


def _read_prefix_plan(ws, lay, S):
    """(header, groups, chunks, others) of a prefix plan in the workspace."""
    hdr = ws[lay["header"]:lay["header"] + 16].view(torch.int32).cpu().tolist()
    ng = max(S // 2, 1)
    groups = ws[lay["groups"]:lay["groups"] + 16 * ng].view(torch.int32).reshape(ng, 4).cpu().tolist()
    chunks = ws[lay["chunks"]:lay["chunks"] + 16 * S].view(torch.int32).reshape(S, 4).cpu().tolist()
    others = ws[lay["others"]:lay["others"] + 4 * S].view(torch.int32).cpu().tolist()
    chunks = chunks[:max(hdr[2], 0)]
    ngroups = max((c[0] for c in chunks), default=-1) + 1   # every group has a chunk
    return hdr, groups[:ngroups], chunks, others[:max(hdr[3], 0)]


def _check_chunks(groups, chunks, nchunks, tiles):
    """Every group's parts 0..parts-1 appear once, as consecutive block ranges
    from 0 to the group's last block, and chunks come in non-increasing work."""
    assert nchunks == sum(g[3] for g in groups)
    assert len(chunks) == nchunks
    seen = {}
    for gi, q, jb, je in chunks:
        seen.setdefault(gi, {})[q] = (jb, je)
    assert sorted(seen) == list(range(len(groups)))
    for gi, (s0, m, P, parts) in enumerate(groups):
        assert 1 <= parts <= 4 and sorted(seen[gi]) == list(range(parts))
        maxn = max(tiles[s0 + k] for k in range(m))
        edges = [seen[gi][q] for q in range(parts)]
        assert edges[0][0] == 0 and edges[-1][1] == maxn
        assert all(edges[q][1] == edges[q + 1][0] for q in range(parts - 1))

    def work(gi, jb, je):
        s0, m, P, _ = groups[gi]
        return max(0, min(je, P) - jb) + sum(max(0, min(je, tiles[s0 + k]) - max(jb, P)) for k in range(m))
    # groups ranked by ceil(work / parts); a group's chunks together
    ranked = [-(-work(gi, 0, 10 ** 9) // groups[gi][3]) for gi, q, _, _ in chunks if q == 0]
    assert ranked == sorted(ranked, reverse=True)


@pytest.mark.parametrize("n,hq,hkv,d,dtype", [(4, 8, 8, 128, "f16"), (3, 16, 8, 64, "bf16"),
                                              (10, 4, 4, 256, "bf16"), (2, 16, 4, 128, "f16")])
def test_shared_prefix_schedule_matches_the_oracle(n, hq, hkv, d, dtype):
    case, trace = _sampling_case(6, n, (70, 300), (0, 40), hq, hkv, d, dtype, seed=n * 7 + d)
    S, mb = case.q.shape[0], case.tables.shape[1]
    assert B.resolved_partition(S, hq, hkv, d, mb, B.SHARED_PREFIX) == B.SHARED_PREFIX
    lay = _prefix_layout(S, hq, hkv, d)
    assert B.workspace_size(S, hq, hkv, d, mb, B.SHARED_PREFIX) == lay["total"]
    ws = torch.full((lay["total"],), 0x3C, dtype=torch.uint8, device="cuda")
    B.paged_attention_plan(case.lens, case.tables, hq, hkv, d, B.SHARED_PREFIX, workspace=ws)
    torch.cuda.synchronize()
    # the plan: each prompt's samples are consecutive sequences; groups of at
    # most 8 / (query heads per KV head) members share the prompt's full
    # blocks (batch order); the rest are the other sequences
    max_members = 8 // (hq // hkv)
    hdr, groups, chunks, others = _read_prefix_plan(ws, lay, S)
    tiles = [-(-L // 16) for L in case.lens.cpu().tolist()]
    want_groups, grouped = [], set()
    for i, P in enumerate(trace.prompt_lens.tolist()):
        if P // 16 < 4:
            continue
        for g0 in range(0, n, max_members):
            m = min(max_members, n - g0)
            if m >= 2:
                want_groups.append([i * n + g0, m, P // 16])
                grouped.update(range(i * n + g0, i * n + g0 + m))
    assert hdr[0] == PREFIX_MAGIC and hdr[1] == S
    assert [g[:3] for g in groups] == want_groups
    assert others == [s for s in range(S) if s not in grouped] and hdr[3] == len(others)
    _check_chunks(groups, chunks, hdr[2], tiles)
    # a grid this small (under one wave) splits its groups into chunks
    assert any(g[3] > 1 for g in groups)
    # two layers with the one plan, then an unplanned call: identical bits, the oracle's values
    outs = []
    for _ in range(2):
        out = case.new_out()
        B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                                 partition_size=B.SHARED_PREFIX, workspace=ws, planned=True)
        outs.append(out)
    plain = _run(case, B.SHARED_PREFIX)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], plain)
    H.assert_attention_close(H.to_f64(outs[0]), H.oracle_full(case), f"shared prefix n={n} {hq}/{hkv} d={d}")
    assert B.device_status(clear=True) == 0


def test_shared_prefix_siblings_with_one_query_are_bit_identical():
    # siblings of one group with equal lengths see the same tiles in the same
    # warps (the others' own tiles are masked out of a row exactly), so with
    # one query for all of them the outputs agree bit for bit
    case, trace = _sampling_case(3, 4, (200, 400), (0, 0), 8, 8, 128, "f16", seed=5)
    q1 = case.q[0:1].expand_as(case.q).contiguous()
    same = H.DecodeCase(q1, case.k_pool, case.v_pool, case.tables, case.lens, case.scale, "f16")
    out = _run(same, B.SHARED_PREFIX)
    n = trace.n
    for i in range(3):
        for c in range(1, n):
            assert torch.equal(out[i * n + c], out[i * n])
    H.assert_attention_close(H.to_f64(out), H.oracle_full(same), "siblings without own tokens")
    assert B.device_status(clear=True) == 0


def test_shared_prefix_without_sharing_is_one_pass_per_sequence():
    # no groups: every sequence in one pass of the tensor-core kernel
    case = H.make_case([37, 300, 1000, 12, 0, 515], 8, 8, 128, "bf16", seed=8)
    out = _run(case, B.SHARED_PREFIX)
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "no sharing")
    assert torch.all(out[4] == 0)
    assert B.device_status(clear=True) == 0


def test_shared_prefix_without_a_plan_is_flagged_and_still_correct():
    case, _ = _sampling_case(4, 4, (100, 200), (1, 30), 8, 8, 64, "f16", seed=9)
    S, mb = case.q.shape[0], case.tables.shape[1]
    ws = torch.full((B.workspace_size(S, 8, 8, 64, mb, B.SHARED_PREFIX),), 0x55, dtype=torch.uint8, device="cuda")
    out = case.new_out()
    B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             partition_size=B.SHARED_PREFIX, workspace=ws, planned=True)
    torch.cuda.synchronize()
    assert B.device_status(clear=True) == 0x20
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "no prefix plan")


def test_shared_prefix_largest_batch():
    # 1024 sequences (the plan kernel's limit: one thread per sequence, up to
    # 512 groups): 256 prompts x 4 samples
    case, _ = _sampling_case(256, 4, (64, 120), (0, 20), 4, 4, 64, "f16", seed=40)
    S, mb = case.q.shape[0], case.tables.shape[1]
    assert S == 1024 and B.resolved_partition(S, 4, 4, 64, mb, B.SHARED_PREFIX) == B.SHARED_PREFIX
    lay = _prefix_layout(S, 4, 4, 64)
    ws = torch.zeros((lay["total"],), dtype=torch.uint8, device="cuda")
    B.paged_attention_plan(case.lens, case.tables, 4, 4, 64, B.SHARED_PREFIX, workspace=ws)
    out = case.new_out()
    B.paged_attention_decode(out, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale,
                             partition_size=B.SHARED_PREFIX, workspace=ws, planned=True)
    torch.cuda.synchronize()
    hdr, groups, chunks, others = _read_prefix_plan(ws, lay, S)
    assert len(groups) == 256 and others == []
    _check_chunks(groups, chunks, hdr[2], [-(-L // 16) for L in case.lens.cpu().tolist()])
    H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "1024 sequences, shared prefix")
    assert B.device_status(clear=True) == 0


def test_shared_prefix_siblings_apart_form_no_groups():
    # the same samples with siblings no longer next to each other: no group
    # forms (sharing that is not consecutive is left to L2) and every
    # sequence runs whole
    case, _ = _sampling_case(6, 4, (100, 300), (0, 40), 8, 8, 128, "bf16", seed=41)
    S = case.q.shape[0]
    perm = torch.from_numpy(np.arange(S).reshape(6, 4).T.reshape(-1).copy()).cuda()  # sibling i of every prompt, in turn
    apart = H.DecodeCase(case.q[perm].contiguous(), case.k_pool, case.v_pool, case.tables[perm].contiguous(),
                         case.lens[perm].contiguous(), case.scale, "bf16")
    lay = _prefix_layout(S, 8, 8, 128)
    ws = torch.zeros((lay["total"],), dtype=torch.uint8, device="cuda")
    B.paged_attention_plan(apart.lens, apart.tables, 8, 8, 128, B.SHARED_PREFIX, workspace=ws)
    torch.cuda.synchronize()
    hdr, groups, chunks, others = _read_prefix_plan(ws, lay, S)
    assert hdr[2] == 0 and others == list(range(S))
    H.assert_attention_close(H.to_f64(_run(apart, B.SHARED_PREFIX)), H.oracle_full(apart), "siblings apart")
    assert B.device_status(clear=True) == 0


def test_shared_prefix_widest_tables():
    # tables of 256 blocks (the widest the plan compares) and a prefix of over
    # 240 shared blocks; a group this long in a grid this small is split
    case, _ = _sampling_case(2, 2, (3900, 4000), (0, 90), 2, 2, 128, "f16", seed=42)
    S, mb = case.q.shape[0], case.tables.shape[1]
    assert mb <= 256
    if mb < 256:   # pad the tables to exactly 256 columns (unused entries -1)
        pad = torch.full((S, 256 - mb), -1, dtype=torch.int32, device="cuda")
        case = H.DecodeCase(case.q, case.k_pool, case.v_pool, torch.cat([case.tables, pad], 1).contiguous(),
                            case.lens, case.scale, "f16")
    lay = _prefix_layout(S, 2, 2, 128)
    ws = torch.zeros((lay["total"],), dtype=torch.uint8, device="cuda")
    B.paged_attention_plan(case.lens, case.tables, 2, 2, 128, B.SHARED_PREFIX, workspace=ws)
    torch.cuda.synchronize()
    hdr, groups, chunks, _ = _read_prefix_plan(ws, lay, S)
    assert len(groups) == 2 and all(g[2] >= 240 and g[3] > 1 for g in groups)
    H.assert_attention_close(H.to_f64(_run(case, B.SHARED_PREFIX)), H.oracle_full(case), "256-block tables")
    assert B.device_status(clear=True) == 0


def test_shared_prefix_full_size_parallel_sampling():
    # the OPT-66B-shaped batch: 32 prompts x 4 samples, 72 heads, head_dim 128
    case, _ = _sampling_case(32, 4, (512, 1024), (0, 256), 72, 72, 128, "f16", seed=21)
    out = _run(case, B.SHARED_PREFIX)
    _check_sampled(case, out, 300, seed=13)
    H.assert_attention_close(H.to_f64(out), H.to_f64(_run(case, -1)), "shared prefix against the grid")
    assert B.device_status(clear=True) == 0
