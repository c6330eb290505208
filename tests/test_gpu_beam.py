"""Beam search and shared prompt prefixes end to end on the GPU: the C++ block
manager drives copy-on-write block copies, cache writes and decode through
the C ABI, the oracle block manager and oracle cache operations do the same
on host copies, and pools and outputs are compared at every step."""

import numpy as np
import pytest
import torch

import helpers as H
import oracle.attention as OA
import oracle.cache_ops as OC
from oracle.block_manager import OracleBlockManager
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


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


@pytest.mark.parametrize("dtype,hq,hkv,d", [("f16", 4, 4, 64), ("bf16", 8, 2, 128)])
def test_beam_search_steps_match_oracle(dtype, hq, hkv, d):
    trace = W.beam_search_trace(seed=3, num_prompts=3, width=3, steps=24, prompt_range=(14, 50),
                                num_heads=hkv, head_dim=d, dtype=dtype)
    nb = trace.block_budget()
    order = W.shuffled_free_order(nb, 5)
    cbm, obm = B.BlockManager(nb, order), OracleBlockManager(nb, initial_free_order=order)
    ids = W.beam_start(trace, cbm)
    assert W.beam_start(trace, obm) == ids
    kp = W.normal_values((nb, hkv, 16, d), dtype, 1, "cuda")
    vp = W.normal_values((nb, hkv, 16, d), dtype, 2, "cuda")
    ok, ov = _bits(kp), _bits(vp)
    mb = -(-(int(trace.prompt_lens.max()) + trace.steps) // 16)
    for step in range(1, trace.steps + 1):
        cs, os_ = W.beam_step(trace, cbm, step), W.beam_step(trace, obm, step)
        assert cs.beam_ids == os_.beam_ids and cs.pairs == os_.pairs
        assert np.array_equal(cs.slots, os_.slots)
        if cs.pairs:
            B.check_copy_pairs(cs.pairs, nb)
            B.copy_blocks(kp, vp, torch.tensor(cs.pairs, dtype=torch.int64, device="cuda"))
            ok, ov = OC.copy_blocks(ok, ov, cs.pairs)
        kn = W.normal_values((len(cs.beam_ids), hkv, d), dtype, 100 + step, "cuda")
        vn = W.normal_values((len(cs.beam_ids), hkv, d), dtype, 200 + step, "cuda")
        B.reshape_and_cache(kn, vn, kp, vp, torch.from_numpy(cs.slots).cuda())
        ok, ov = OC.reshape_and_cache(_bits(kn), _bits(vn), ok, ov, cs.slots)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(kp), ok) and np.array_equal(_bits(vp), ov), f"pools differ at step {step}"
        tables, lens = cbm.block_tables(cs.beam_ids, mb)
        rows, olens = obm.padded_tables(cs.beam_ids, mb)
        assert tables.tolist() == rows and lens.tolist() == olens
        q = W.normal_values((len(cs.beam_ids), hq, d), dtype, 300 + step, "cuda")
        case = H.DecodeCase(q, kp, vp, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                            d ** -0.5, dtype)
        out = case.new_out()
        B.paged_attention_decode(out, q, kp, vp, case.tables, case.lens, case.scale)
        torch.cuda.synchronize()
        H.assert_attention_close(H.to_f64(out), H.oracle_full(case), f"step {step}")
    assert B.device_status(clear=True) == 0


def test_full_size_beam_search_sampled():
    trace = W.beam_search_trace(0)
    nb = trace.block_budget()
    bm = B.BlockManager(nb, W.shuffled_free_order(nb, 0))
    W.beam_start(trace, bm)
    hkv, d = trace.num_kv_heads, trace.head_dim
    kp = W.normal_values((nb, hkv, 16, d), "bf16", 1, "cuda")
    vp = W.normal_values((nb, hkv, 16, d), "bf16", 2, "cuda")
    for step in range(1, trace.steps + 1):
        st = W.beam_step(trace, bm, step)
        if st.pairs:
            B.copy_blocks(kp, vp, torch.tensor(st.pairs, dtype=torch.int64, device="cuda"))
        kn = W.normal_values((len(st.beam_ids), hkv, d), "bf16", 10 + step, "cuda")
        B.reshape_and_cache(kn, kn, kp, vp, torch.from_numpy(st.slots).cuda())
    mb = -(-(int(trace.prompt_lens.max()) + trace.steps) // 16)
    tables, lens = bm.block_tables(st.beam_ids, mb)
    q = W.normal_values((len(st.beam_ids), trace.num_q_heads, d), "bf16", 3, "cuda")
    case = H.DecodeCase(q, kp, vp, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                        trace.scale, "bf16")
    rng = np.random.default_rng(4)
    S = len(st.beam_ids)
    pairs = sorted({(int(s), int(h)) for s, h in zip(rng.integers(0, S, 16), rng.integers(0, trace.num_q_heads, 16))}
                   | {(s, int(h)) for s, h in zip(range(S), rng.integers(0, trace.num_q_heads, S))})
    want = H.oracle_sampled(case, pairs)
    # the default schedule, and the shared-prefix schedule (beams of a prompt
    # grouped; few groups, so each group's work is split over several CTAs)
    outs = []
    for partition in (0, B.SHARED_PREFIX):
        out = case.new_out()
        B.paged_attention_decode(out, q, kp, vp, case.tables, case.lens, case.scale, partition_size=partition)
        torch.cuda.synchronize()
        got = H.to_f64(out)
        for (s, h), w in want.items():
            H.assert_attention_close(got[s, h], w, f"partition {partition}: beam {s} head {h}")
        outs.append(got)
    H.assert_attention_close(outs[1], outs[0], "shared prefix against the default schedule")
    # beams share most of their blocks: far fewer unique blocks than table entries
    used = tables[tables >= 0]
    assert np.unique(used).size < 0.5 * used.size
    assert B.device_status(clear=True) == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_shared_prefix_requests(dtype):
    # a donor request holds a 70-token system prompt; three requests repeat the
    # first 70 tokens and go on with their own; only whole blocks are shared,
    # and the result equals that of private copies of the same tokens
    hkv, hq, d, nb = 4, 8, 128, 64
    bm = B.BlockManager(nb, W.shuffled_free_order(nb, 2))
    private = B.BlockManager(nb, W.shuffled_free_order(nb, 9))
    kp = W.normal_values((nb, hkv, 16, d), dtype, 5, "cuda")
    vp = W.normal_values((nb, hkv, 16, d), dtype, 6, "cuda")
    kp2, vp2 = kp.clone(), vp.clone()
    prompt = W.normal_values((70, hkv, d), dtype, 7, "cuda"), W.normal_values((70, hkv, d), dtype, 8, "cuda")
    lens = [70, 95, 80, 150]
    toks = [prompt] + [(torch.cat([prompt[0], W.normal_values((L - 70, hkv, d), dtype, 20 + i, "cuda")]),
                        torch.cat([prompt[1], W.normal_values((L - 70, hkv, d), dtype, 30 + i, "cuda")]))
                       for i, L in enumerate(lens[1:])]
    bm.add_seq(0, 70)
    private.add_seq(0, 70)
    starts = [0]
    for s, L in enumerate(lens[1:], start=1):
        starts.append(bm.add_seq_with_prefix(s, L, 0, 70))
        private.add_seq(s, L)
    assert starts == [0, 64, 64, 64]

    def write(mgr, k_pool, v_pool, first):
        for s, (k, v) in enumerate(toks):
            t, _ = mgr.block_tables([s], 16)
            pos = np.arange(first[s], lens[s])
            slots = t[0, pos // 16].astype(np.int64) * 16 + pos % 16
            B.reshape_and_cache(k[first[s]:].contiguous(), v[first[s]:].contiguous(), k_pool, v_pool,
                                torch.from_numpy(slots).cuda())

    write(bm, kp, vp, starts)
    write(private, kp2, vp2, [0] * 4)
    q = W.normal_values((4, hq, d), dtype, 9, "cuda")
    outs = []
    for mgr, k_pool, v_pool in ((bm, kp, vp), (private, kp2, vp2)):
        tables, L = mgr.block_tables(range(4), 16)
        case = H.DecodeCase(q, k_pool, v_pool, torch.from_numpy(tables).cuda(), torch.from_numpy(L).cuda(),
                            d ** -0.5, dtype)
        out = case.new_out()
        B.paged_attention_decode(out, q, k_pool, v_pool, case.tables, case.lens, case.scale)
        torch.cuda.synchronize()
        H.assert_attention_close(H.to_f64(out), H.oracle_full(case), "prefix")
        outs.append(out)
    assert torch.equal(outs[0], outs[1])           # sharing changes where data lives, not the result
    assert bm.num_free() == private.num_free() + 3 * 4   # four whole prompt blocks shared by three requests
    assert B.device_status(clear=True) == 0
