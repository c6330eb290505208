"""GPU parity of sliding-window decode (through the C ABI) against the oracle:
each query attends over its sequence's last W tokens; table entries before
the window (released by the block manager) are never read."""

import numpy as np
import pytest
import torch

import helpers as H
import oracle.attention as OA
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


def _oracle_window(case, window, tables=None):
    t = case.tables if tables is None else tables
    return OA.paged_attention_decode_window(
        W.to_numpy_storage(case.q, case.dtype), W.to_numpy_storage(case.k_pool, case.dtype),
        W.to_numpy_storage(case.v_pool, case.dtype), t.cpu().numpy(), case.lens.cpu().numpy(),
        case.scale, case.num_kv_heads, case.dtype, window)


def _run(case, window, partition=0, tables=None):
    out = case.new_out()
    B.paged_attention_decode_sliding(out, case.q, case.k_pool, case.v_pool,
                                     case.tables if tables is None else tables, case.lens, case.scale, window,
                                     partition_size=partition)
    torch.cuda.synchronize()
    return out


def _release(tables, lens, window):
    """Tables with every entry wholly before each sequence's window set to -1."""
    t = tables.clone()
    for s, L in enumerate(lens.tolist()):
        first = OA.window_start(L, window)
        t[s, :first // 16] = -1
    return t


RAGGED = [0, 1, 15, 16, 17, 33, 100, 257, 530]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (8, 8, 128), (2, 2, 256), (8, 2, 128), (16, 2, 64),
                                      (8, 1, 256)])
@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 4096])
def test_sliding_parity(dtype, hq, hkv, d, window):
    case = H.make_case(RAGGED, hq, hkv, d, dtype, seed=hq + d + window, extra_cols=1)
    want = _oracle_window(case, window)
    got = H.to_f64(_run(case, window))
    H.assert_attention_close(got, want, f"{dtype} hq={hq} hkv={hkv} d={d} W={window}")
    assert np.all(got[0] == 0.0)
    assert B.device_status(clear=True) == 0


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 8)])
@pytest.mark.parametrize("partition", [0, -1, 16, 48, 256])
def test_sliding_schedules(hq, hkv, partition):
    case = H.make_case([700, 31, 1000, 4, 513, 64], hq, hkv, 128, "bf16", seed=5)
    for window in (33, 200, 512):
        want = _oracle_window(case, window)
        H.assert_attention_close(H.to_f64(_run(case, window, partition)), want,
                                 f"hq={hq} partition={partition} W={window}")
    assert B.device_status(clear=True) == 0


@pytest.mark.parametrize("hq,hkv", [(4, 4), (16, 4)])
def test_released_entries_are_never_read(hq, hkv):
    case = H.make_case([600, 37, 250, 1024], hq, hkv, 128, "f16", seed=7)
    for window in (1, 40, 129):
        t = _release(case.tables, case.lens.cpu(), window).to(case.tables.device)
        want = _oracle_window(case, window, t)
        for partition in (0, -1, 64):
            H.assert_attention_close(H.to_f64(_run(case, window, partition, t)), want, f"W={window}")
        assert B.device_status(clear=True) == 0      # no -1 entry was read


def test_no_window_is_full_decode():
    case = H.make_case(RAGGED, 8, 4, 128, "bf16", seed=9)
    full = case.new_out()
    B.paged_attention_decode(full, case.q, case.k_pool, case.v_pool, case.tables, case.lens, case.scale)
    torch.cuda.synchronize()
    for window in (0, -5, 530, 10_000):
        assert torch.equal(_run(case, window), full)


def test_long_context_window():
    case = H.make_case([9000, 20000, 4100, 16384], 16, 8, 128, "bf16", seed=11)
    lens = case.lens.cpu().numpy()
    rng = np.random.default_rng(1)
    for window in (4096, 4111):
        got = _run(case, window)
        pairs = [(int(s), int(h)) for s, h in zip(rng.integers(0, 4, 6), rng.integers(0, 16, 6))]
        for s, h in pairs:
            # the oracle on just this (sequence, head) with its window
            g = h // 2
            L = int(lens[s])
            first = OA.window_start(L, window)
            b0, b1 = first // 16, -(-L // 16)
            ids = case.tables[s, b0:b1].long()
            kp = case.k_pool[:, g].index_select(0, ids).unsqueeze(1)
            vp = case.v_pool[:, g].index_select(0, ids).unsqueeze(1)
            sub_t = np.arange(b1 - b0, dtype=np.int32).reshape(1, -1)
            want = OA.paged_attention_decode_window(
                W.to_numpy_storage(case.q[s, h].reshape(1, 1, -1), "bf16"), W.to_numpy_storage(kp, "bf16"),
                W.to_numpy_storage(vp, "bf16"), sub_t, np.array([L - 16 * b0], np.int32), case.scale, 1, "bf16",
                window)
            H.assert_attention_close(H.to_f64(got[s, h]), want[0, 0], f"W={window} ({s}, {h})")
    assert B.device_status(clear=True) == 0


def test_decode_steps_with_block_release():
    # a block-manager-driven run: each step writes the new token, releases
    # blocks before the window and decodes; the free list grows back as the
    # window slides
    window, hkv, hq, d, dtype = 40, 2, 4, 64, "f16"
    nb = 64
    order = W.shuffled_free_order(nb, 3)
    bm = B.BlockManager(nb, order)
    prompts = [30, 70, 5]
    for s, L in enumerate(prompts):
        bm.add_seq(s, L)
    k_pool = W.normal_values((nb, hkv, 16, d), dtype, 1, "cuda")
    v_pool = W.normal_values((nb, hkv, 16, d), dtype, 2, "cuda")
    for step in range(40):
        slots, pairs = bm.append_slots(range(3))
        assert pairs.shape[0] == 0
        knew = W.normal_values((3, hkv, d), dtype, 100 + step, "cuda")
        vnew = W.normal_values((3, hkv, d), dtype, 200 + step, "cuda")
        B.reshape_and_cache(knew, vnew, k_pool, v_pool, torch.from_numpy(slots).cuda())
        for s in range(3):
            bm.release_before(s, OA.window_start(bm.seq_len(s), window))
        tables, lens = bm.block_tables(range(3), 8)
        q = W.normal_values((3, hq, d), dtype, 300 + step, "cuda")
        out = torch.empty_like(q)
        tt, ll = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
        B.paged_attention_decode_sliding(out, q, k_pool, v_pool, tt, ll, d ** -0.5, window)
        torch.cuda.synchronize()
        want = OA.paged_attention_decode_window(
            W.to_numpy_storage(q, dtype), W.to_numpy_storage(k_pool, dtype), W.to_numpy_storage(v_pool, dtype),
            tables, lens, d ** -0.5, hkv, dtype, window)
        H.assert_attention_close(H.to_f64(out), want, f"step {step}")
        live = sum(1 for s in range(3) for b in bm.block_table(s) if b >= 0)
        assert bm.num_free() == nb - live
        assert all(sum(1 for b in bm.block_table(s) if b >= 0) <= -(-window // 16) + 1 for s in range(3))
    assert B.device_status(clear=True) == 0


def test_balanced_schedule_rejects_a_window():
    case = H.make_case([20, 30], 8, 8, 128, "bf16", seed=4)
    with pytest.raises(B.PagedKVError) as ei:
        _run(case, 16, B.BALANCED)
    assert ei.value.status == 2


def test_sliding_window_with_batch_ranked_once():
    # 140 sequences: the ordering kernel ranks by the windowed lengths
    rng = np.random.default_rng(3)
    lens = rng.integers(1, 80, 140).astype(np.int32)
    lens[[5, 60]] = [1000, 600]
    case = H.make_case(lens, 8, 2, 64, "bf16", seed=23)
    for window in (16, 100):
        want = _oracle_window(case, window)
        H.assert_attention_close(H.to_f64(_run(case, window)), want, f"W={window}")
    assert B.device_status(clear=True) == 0
