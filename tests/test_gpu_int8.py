"""GPU parity of the INT8 KV cache (through the C ABI) against the oracle:
quantising cache write and block copies bit-exact (codes and scales), decode
over the INT8 cache within the attention tolerance."""

import numpy as np
import pytest
import torch

import helpers as H
import oracle.cache_ops as OC
import oracle.quant as OQ
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


def _np(t):
    return t.detach().cpu().contiguous().numpy()


def _int8_cache(nb, hkv, d, seed, device="cuda"):
    kc = W.int8_codes((nb, hkv, 16, d), seed * 5 + 1, device)
    vc = W.int8_codes((nb, hkv, 16, d), seed * 5 + 2, device)
    ks = W.row_scales((nb, hkv, 16), seed * 5 + 3, device)
    vs = W.row_scales((nb, hkv, 16), seed * 5 + 4, device)
    return kc, vc, ks, vs


# ---- quantising cache write ---------------------------------------------------
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hkv,d", [(4, 64), (8, 128), (2, 256), (40, 128)])
def test_reshape_int8_bit_exact(dtype, hkv, d):
    nb, T = 30, 101
    rng = np.random.default_rng(hkv * 1000 + d)
    slots = rng.choice(nb * 16, size=T, replace=False).astype(np.int64)
    slots[::9] = -1                                        # skipped tokens
    kc, vc, ks, vs = _int8_cache(nb, hkv, d, 3)
    k = W.normal_values((T, hkv, d), dtype, 11, "cuda")
    v = W.normal_values((T, hkv, d), dtype, 12, "cuda")
    k[5] = 0                                               # all-zero rows: scale 0, codes 0
    v[6, 1 % hkv] = 0
    before = [_np(x) for x in (kc, vc, ks, vs)]
    B.reshape_and_cache_int8(k, v, kc, vc, ks, vs, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    want = OQ.reshape_and_cache_int8(W.to_numpy_storage(k, dtype), W.to_numpy_storage(v, dtype), dtype,
                                     *before, slots)
    for got, exp, name in zip((kc, vc, ks, vs), want, ("k codes", "v codes", "k scales", "v scales")):
        g = _np(got)
        if g.dtype == np.float32:   # scales compared as bit patterns
            g, exp = g.view(np.uint32), np.asarray(exp, np.float32).view(np.uint32)
        assert np.array_equal(g, exp), f"{name} differ at {np.argwhere(g != exp)[:5].tolist()}"
    assert B.device_status(clear=True) == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_reshape_int8_ties_round_to_even(dtype):
    # max |x| = 127 gives s = 1 exactly, so x / s = x: halves are ties
    d, hkv = 64, 1
    row = np.zeros(d, np.float32)
    row[:8] = [127.0, 2.5, -3.5, 0.5, -0.5, 1.5, 126.5, -125.5]
    k = torch.from_numpy(np.stack([row])[:, None, :]).to(H.torch_dtype(dtype)).cuda()
    v = (-k).contiguous()
    kc, vc, ks, vs = _int8_cache(2, hkv, d, 4)
    B.reshape_and_cache_int8(k, v, kc, vc, ks, vs, torch.tensor([17], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert float(ks[1, 0, 1]) == 1.0 and float(vs[1, 0, 1]) == 1.0
    assert _np(kc[1, 0, 1, :8]).tolist() == [127, 2, -4, 0, 0, 2, 126, -126]
    assert _np(vc[1, 0, 1, :8]).tolist() == [-127, -2, 4, 0, 0, -2, -126, 126]


def test_reshape_int8_bad_slot_flagged():
    d, hkv, nb = 128, 2, 4
    kc, vc, ks, vs = _int8_cache(nb, hkv, d, 5)
    before = [_np(x) for x in (kc, vc, ks, vs)]
    k = W.normal_values((2, hkv, d), "bf16", 1, "cuda")
    B.reshape_and_cache_int8(k, k.clone(), kc, vc, ks, vs,
                             torch.tensor([nb * 16, nb * 16 + 5], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert B.device_status(clear=True) & 0x4
    for got, exp in zip((kc, vc, ks, vs), before):
        assert np.array_equal(_np(got), exp)


# ---- block copies ----------------------------------------------------------------
def test_copy_blocks_int8_bit_exact():
    nb, hkv, d = 24, 8, 128
    kc, vc, ks, vs = _int8_cache(nb, hkv, d, 6)
    pairs = np.array([[0, 5], [3, 7], [3, 9], [20, 1]], np.int64)
    B.check_copy_pairs(pairs, nb)
    before = [_np(x) for x in (kc, vc, ks, vs)]
    B.copy_blocks_int8(kc, vc, ks, vs, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    ekc, evc = OC.copy_blocks(before[0], before[1], pairs)
    eks, evs = OC.copy_blocks(before[2], before[3], pairs)
    for got, exp in zip((kc, vc, ks, vs), (ekc, evc, eks, evs)):
        assert np.array_equal(_np(got), exp)
    assert B.device_status(clear=True) == 0


# ---- decode over the INT8 cache ---------------------------------------------------
class Int8Case:
    def __init__(self, lens, hq, hkv, d, dtype, seed, extra_cols=0):
        lens = np.asarray(lens, np.int32)
        nb = W.pool_size(lens, 1.2) + 1
        tables, _ = W.scattered_tables(lens, nb, seed, extra_cols=extra_cols)
        self.kc, self.vc, self.ks, self.vs = _int8_cache(nb, hkv, d, seed)
        self.q = W.normal_values((len(lens), hq, d), dtype, seed * 5 + 7, "cuda")
        self.tables = torch.from_numpy(tables).cuda()
        self.lens = torch.from_numpy(lens).cuda()
        self.scale = d ** -0.5
        self.dtype, self.hkv = dtype, hkv

    def run(self, partition_size=0):
        out = torch.full_like(self.q, float("nan"))
        B.paged_attention_decode_int8(out, self.q, self.kc, self.vc, self.ks, self.vs, self.tables, self.lens,
                                      self.scale, partition_size=partition_size)
        torch.cuda.synchronize()
        return out

    def oracle(self):
        return OQ.paged_attention_decode_int8(
            W.to_numpy_storage(self.q, self.dtype), _np(self.kc), _np(self.vc), _np(self.ks), _np(self.vs),
            _np(self.tables), _np(self.lens), self.scale, self.hkv, self.dtype)

    def oracle_rows(self, pairs):
        """Oracle rows for a few (seq, q head) pairs, each over a sub-pool of
        the blocks its sequence uses (relabelled ids)."""
        group = self.q.shape[1] // self.hkv
        lens, tables = _np(self.lens), _np(self.tables)
        rows = {}
        for s, h in pairs:
            g, L = h // group, int(lens[s])
            nb = -(-L // 16)
            ids = torch.from_numpy(tables[s, :max(nb, 1)].astype(np.int64)).cuda()
            sub = [x[:, g].index_select(0, ids).unsqueeze(1) for x in (self.kc, self.vc, self.ks, self.vs)]
            out = OQ.paged_attention_decode_int8(
                W.to_numpy_storage(self.q[s, h].reshape(1, 1, -1), self.dtype), *[_np(x) for x in sub],
                np.arange(max(nb, 1), dtype=np.int32).reshape(1, -1), np.array([L], np.int32), self.scale, 1,
                self.dtype)
            rows[(s, h)] = out[0, 0]
        return rows


RAGGED = [0, 1, 15, 16, 17, 33, 100, 257, 530]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (8, 8, 128), (2, 2, 256), (8, 4, 128), (16, 4, 64),
                                      (16, 2, 128), (8, 1, 256), (12, 2, 128)])
@pytest.mark.parametrize("partition", [0, -1, 64])
def test_decode_int8_parity(dtype, hq, hkv, d, partition):
    case = Int8Case(RAGGED, hq, hkv, d, dtype, seed=hq + d, extra_cols=2)
    got = H.to_f64(case.run(partition))
    H.assert_attention_close(got, case.oracle(), f"int8 {dtype} hq={hq} hkv={hkv} d={d} p={partition}")
    assert np.all(got[0] == 0.0)                            # empty sequence gives zeros
    assert B.device_status(clear=True) == 0


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 128), (4, 4, 64), (4, 1, 256)])
@pytest.mark.parametrize("partition", [0, 16])
def test_decode_int8_every_partial_tile_size(hq, hkv, d, partition):
    # lengths 1..48: the last code tile of a sequence (or of a split part)
    # holds every count of valid rows from 1 to 16, copied as boxes of 16, 8
    # and 4 rows
    case = Int8Case(np.arange(1, 49), hq, hkv, d, "bf16", seed=70 + d)
    got = H.to_f64(case.run(partition))
    H.assert_attention_close(got, case.oracle(), f"int8 partial tiles hq={hq} hkv={hkv} d={d} p={partition}")
    assert B.device_status(clear=True) == 0


def test_decode_int8_split_partitions_long():
    # several partitions per sequence, the last one ragged, with the default schedule and explicit ones
    case = Int8Case([3000, 2049, 17, 4096], 16, 8, 128, "bf16", seed=21)
    want = case.oracle()
    for p in (0, 256, 512, -1):
        H.assert_attention_close(H.to_f64(case.run(p)), want, f"partition {p}")
    assert B.device_status(clear=True) == 0


def test_decode_int8_zero_scale_rows():
    # rows stored as all-zero (scale 0) take part in the softmax with score 0
    case = Int8Case([40, 64], 4, 4, 64, "f16", seed=3)
    case.ks[:, :, 3] = 0
    case.vs[:, :, 5] = 0
    H.assert_attention_close(H.to_f64(case.run()), case.oracle(), "zero-scale rows")


def test_decode_int8_balanced_rejected():
    case = Int8Case([20, 30], 8, 8, 128, "bf16", seed=4)
    with pytest.raises(B.PagedKVError) as ei:
        case.run(B.BALANCED)
    assert ei.value.status == 2


@pytest.mark.parametrize("name", ["llama13b", "llama3_8b", "opt175b"])
def test_decode_int8_full_size_sampled(name):
    # the OPT-175B layer (768 CTAs of 16-32k tokens) runs the 8-warp one-query
    # tile, whose warps walk more than 32 blocks of ids each
    shape = {"llama13b": W.llama13b_mha_decode, "llama3_8b": W.llama3_8b_gqa_decode,
             "opt175b": W.opt175b_long_decode}[name](0)
    case = Int8Case(shape.context_lens, shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.dtype,
                    seed=1)
    got = case.run()
    S, Hq = case.q.shape[0], case.q.shape[1]
    rng = np.random.default_rng(7)
    pairs = [(int(s), int(h)) for s, h in zip(rng.integers(0, S, 12), rng.integers(0, Hq, 12))]
    pairs.append((int(np.argmax(shape.context_lens)), Hq - 1))
    rows = case.oracle_rows(pairs)
    for (s, h), want in rows.items():
        H.assert_attention_close(H.to_f64(got[s, h]), want, f"{name} int8 ({s}, {h})")
    assert torch.isfinite(got.float()).all()
    assert B.device_status(clear=True) == 0


def test_decode_int8_large_v_rows_on_the_tensor_cores():
    # V rows whose dequantised values exceed the fp16 range (possible for bf16
    # inputs): the V scale rides on the softmax weight (with a power of two per
    # warp), the codes stay exact in fp16, so nothing overflows
    big = Int8Case([40, 300, 17], 4, 4, 128, "bf16", seed=91)
    big.vc.fill_(100)
    big.vs.mul_(65536.0)
    want = big.oracle()
    assert np.abs(want).max() > 65504.0
    H.assert_attention_close(H.to_f64(big.run()), want, "int8 large V rows")
    assert B.device_status(clear=True) == 0


def test_decode_int8_v_scales_spanning_many_magnitudes():
    # scales from 2^-30 to 2^20 in random blocks: the warps' power of two falls
    # tile after tile and the accumulator is rescaled with it (bf16 outputs:
    # values past the fp16 range stay finite)
    case = Int8Case([700, 1200, 33, 16, 2000], 8, 2, 128, "bf16", seed=92)
    rng = np.random.default_rng(5)
    nb = case.vs.shape[0]
    mags = torch.from_numpy(np.exp2(rng.integers(-30, 21, size=(nb, 1, 1))).astype(np.float32)).cuda()
    case.vs.mul_(mags)
    case.ks.mul_(torch.from_numpy(np.exp2(rng.integers(-3, 4, size=(nb, 1, 1))).astype(np.float32)).cuda())
    want = case.oracle()
    # Each weight enters the tensor cores as one fp16 value (11 significant
    # bits), so an output element that is a near-cancelling sum of terms up to
    # 2^27 carries an error of ~2^-11 of those terms, not of itself: the bound
    # is taken against the largest output of its row (a lost rescale or an
    # overflow would be off by the whole row).
    row_max = np.abs(want).max(axis=-1, keepdims=True)
    for p in (0, -1, 64):
        got = H.to_f64(case.run(p))
        assert np.all(np.isfinite(got)), p
        assert np.all(np.abs(got - want) <= 2e-3 * row_max + 1e-2 * np.abs(want)), \
            (p, float(np.max(np.abs(got - want) / row_max)))
    assert B.device_status(clear=True) == 0


def test_decode_int8_planned():
    # the step's launch plan (made by paged_attention_plan, shared with the
    # 16-bit cache) used by the planned INT8 entry point; a workspace holding
    # no plan flags BAD_PLAN and still computes every output
    rng = np.random.default_rng(8)
    lens = np.clip(np.round(150 * np.exp(0.6 * rng.standard_normal(200))), 8, 1024).astype(np.int32)
    case = Int8Case(lens, 32, 8, 128, "bf16", seed=93)
    S, mb = case.q.shape[0], case.tables.shape[1]
    ws = torch.zeros((B.workspace_size(S, 32, 8, 128, mb),), dtype=torch.uint8, device="cuda")
    B.paged_attention_plan(case.lens, case.tables, 32, 8, 128, workspace=ws)
    want = case.oracle()
    for planned_ws in (ws, torch.zeros_like(ws)):
        out = torch.full_like(case.q, float("nan"))
        B.paged_attention_decode_int8(out, case.q, case.kc, case.vc, case.ks, case.vs, case.tables, case.lens,
                                      case.scale, workspace=planned_ws, planned=True)
        torch.cuda.synchronize()
        H.assert_attention_close(H.to_f64(out), want, "planned int8")
        assert B.device_status(clear=True) == (0 if planned_ws is ws else 0x20)


# ---- the shared-prefix schedule over the INT8 cache ----------------------------------
def _int8_sampling_case(num_prompts, n, prompt_range, tail_range, hq, hkv, d, dtype, seed):
    """Tables of parallel samples from the block manager (prompt added, forked
    n-1 times, tails appended with copy-on-write) over a random INT8 cache."""
    trace = W.ParallelSamplingTrace("sampling", dtype, hq, hkv, d,
                                    np.random.default_rng(seed).integers(*prompt_range, size=num_prompts,
                                                                         endpoint=True).astype(np.int32),
                                    np.random.default_rng(seed + 1).integers(*tail_range, size=(num_prompts, n),
                                                                             endpoint=True).astype(np.int32))
    nb = trace.block_budget()
    bm = B.BlockManager(nb, W.shuffled_free_order(nb, seed))
    plan = W.drive_parallel_sampling(trace, bm)
    mb = max(-(-L // 16) for L in plan.final_lens.values())
    tables, lens = bm.block_tables(plan.seq_ids, mb)
    case = Int8Case.__new__(Int8Case)
    case.kc, case.vc, case.ks, case.vs = _int8_cache(nb, hkv, d, seed)
    case.q = W.normal_values((len(plan.seq_ids), hq, d), dtype, seed * 5 + 7, "cuda")
    case.tables = torch.from_numpy(tables).cuda()
    case.lens = torch.from_numpy(lens).cuda()
    case.scale = d ** -0.5
    case.dtype, case.hkv = dtype, hkv
    return case, trace


@pytest.mark.parametrize("n,hq,hkv,d,dtype", [(4, 8, 8, 128, "f16"), (3, 16, 8, 64, "bf16"),
                                              (10, 4, 4, 256, "bf16"), (2, 16, 4, 128, "f16")])
def test_decode_int8_shared_prefix_matches_the_oracle(n, hq, hkv, d, dtype):
    # small batches: the plan splits groups into chunks merged by log-sum-exp
    case, _ = _int8_sampling_case(6, n, (70, 300), (0, 40), hq, hkv, d, dtype, seed=n * 7 + d)
    want = case.oracle()
    got = case.run(B.SHARED_PREFIX)
    H.assert_attention_close(H.to_f64(got), want, f"int8 shared prefix n={n} {hq}/{hkv} d={d}")
    H.assert_attention_close(H.to_f64(case.run(0)), want, "int8 default schedule")
    assert B.device_status(clear=True) == 0


def test_decode_int8_shared_prefix_siblings_are_bit_identical():
    case, trace = _int8_sampling_case(3, 4, (200, 400), (0, 0), 8, 8, 128, "f16", seed=5)
    case.q = case.q[0:1].expand_as(case.q).contiguous()
    out = case.run(B.SHARED_PREFIX)
    n = trace.n
    for i in range(3):
        for c in range(1, n):
            assert torch.equal(out[i * n + c], out[i * n])
    H.assert_attention_close(H.to_f64(out), case.oracle(), "int8 siblings")
    assert B.device_status(clear=True) == 0


def test_decode_int8_shared_prefix_planned_and_unplanned():
    case, _ = _int8_sampling_case(5, 4, (100, 260), (1, 30), 8, 8, 64, "bf16", seed=9)
    S, mb = case.q.shape[0], case.tables.shape[1]
    want = case.oracle()
    ws = torch.full((B.workspace_size(S, 8, 8, 64, mb, B.SHARED_PREFIX),), 0x55, dtype=torch.uint8, device="cuda")
    # no plan in the workspace: flagged, every sequence whole
    out = torch.full_like(case.q, float("nan"))
    B.paged_attention_decode_int8(out, case.q, case.kc, case.vc, case.ks, case.vs, case.tables, case.lens,
                                  case.scale, partition_size=B.SHARED_PREFIX, workspace=ws, planned=True)
    torch.cuda.synchronize()
    assert B.device_status(clear=True) == 0x20
    H.assert_attention_close(H.to_f64(out), want, "int8 shared prefix without a plan")
    # the plan of the 16-bit call serves the INT8 call; two layers with it
    B.paged_attention_plan(case.lens, case.tables, 8, 8, 64, B.SHARED_PREFIX, workspace=ws)
    outs = []
    for _ in range(2):
        out = torch.full_like(case.q, float("nan"))
        B.paged_attention_decode_int8(out, case.q, case.kc, case.vc, case.ks, case.vs, case.tables, case.lens,
                                      case.scale, partition_size=B.SHARED_PREFIX, workspace=ws, planned=True)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    H.assert_attention_close(H.to_f64(outs[0]), want, "int8 shared prefix planned")
    assert B.device_status(clear=True) == 0


def test_decode_int8_shared_prefix_full_size_sampling():
    # the OPT-66B-shaped batch: 32 prompts x 4 samples, 72 heads, head_dim 128
    case, _ = _int8_sampling_case(32, 4, (512, 1024), (0, 256), 72, 72, 128, "f16", seed=21)
    got = case.run(B.SHARED_PREFIX)
    S, Hq = case.q.shape[0], case.q.shape[1]
    rng = np.random.default_rng(13)
    pairs = sorted({(s, int(h)) for s, h in zip(range(S), rng.integers(0, Hq, S))})
    rows = case.oracle_rows(pairs)
    for (s, h), want in rows.items():
        H.assert_attention_close(H.to_f64(got[s, h]), want, f"int8 shared prefix ({s}, {h})")
    H.assert_attention_close(H.to_f64(got), H.to_f64(case.run(-1)), "int8 shared prefix against one pass")
    assert B.device_status(clear=True) == 0


# ---- the CUDA-core INT8 tile (a build with PKV_INT8_MMA=0) -------------------------
@pytest.fixture(scope="module")
def cuda_core_int8_lib(tmp_path_factory):
    """The library built with the CUDA-core INT8 tile (codes to fp32 exactly, the
    K scale on the reduced score, the V scale folded into the softmax weight),
    loaded in place of the default build for the tests that take it."""
    from paged_kv_cache_217_gb300 import build
    path = build.build(out_dir=str(tmp_path_factory.mktemp("int8_cuda_core")), defines=["PKV_INT8_MMA=0"])
    saved = (B.LIB_PATH, B._lib)
    B.LIB_PATH, B._lib = path, None
    try:
        B.lib()
        yield path
    finally:
        B.LIB_PATH, B._lib = saved


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (8, 8, 128), (8, 2, 128), (8, 1, 256)])
@pytest.mark.parametrize("partition", [0, -1, 64])
def test_cuda_core_int8_tile_parity(cuda_core_int8_lib, dtype, hq, hkv, d, partition):
    case = Int8Case(RAGGED, hq, hkv, d, dtype, seed=hq + d + 1, extra_cols=2)
    got = H.to_f64(case.run(partition))
    H.assert_attention_close(got, case.oracle(), f"cuda-core int8 {dtype} hq={hq} hkv={hkv} d={d} p={partition}")
    assert np.all(got[0] == 0.0)
    assert B.device_status(clear=True) == 0


def test_cuda_core_int8_tile_partial_tiles_and_large_rows(cuda_core_int8_lib):
    case = Int8Case(np.arange(1, 49), 8, 2, 128, "bf16", seed=90)
    H.assert_attention_close(H.to_f64(case.run(16)), case.oracle(), "cuda-core int8 partial tiles")
    # V rows whose dequantised values exceed the fp16 range (possible for bf16
    # inputs): the CUDA-core tile keeps them in fp32
    big = Int8Case([40, 300, 17], 4, 4, 128, "bf16", seed=91)
    big.vc.fill_(100)
    big.vs.mul_(65536.0)
    want = big.oracle()
    assert np.abs(want).max() > 65504.0
    H.assert_attention_close(H.to_f64(big.run()), want, "cuda-core int8 large V rows")
    assert B.device_status(clear=True) == 0


def test_cuda_core_int8_tile_has_no_shared_prefix_schedule(cuda_core_int8_lib):
    case, _ = _int8_sampling_case(2, 4, (100, 200), (0, 10), 8, 8, 128, "bf16", seed=94)
    with pytest.raises(B.PagedKVError) as ei:
        case.run(B.SHARED_PREFIX)
    assert ei.value.status == 2
