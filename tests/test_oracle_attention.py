"""Pins of the fp64 attention oracle against facts that do not come from the oracle.

* hand-worked values (tests/golden/one_block_example.json),
* brute force on tiny inputs: dense per-token Python loops with math.exp,
  written without block tables, numpy or the oracle's helpers,
* closed forms: L=1 gives v0 exactly, equal keys or q=0 give the mean of V,
  GQA groups with constant V per KV head,
* invariance of the output under relabelling physical blocks
  (the block table makes placement irrelevant),
* the log-sum-exp merge of partition pieces equals the unsplit softmax,
* planted mistakes in a copy of the oracle are each caught by some pin.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import attention as OA
from oracle.numerics import to_f64, round_to

BS = 16


def _f16(x):
    return np.asarray(x, dtype=np.float16)


def _pool_from_dense(dense_per_head, lengths, tables, num_blocks, head_dim, fill=0.0):
    """Scatter dense [Hkv][s][L_s][d] data into a [num_blocks, Hkv, 16, d] pool."""
    hkv = len(dense_per_head)
    pool = np.full((num_blocks, hkv, BS, head_dim), fill, dtype=np.float16)
    for g in range(hkv):
        for s, L in enumerate(lengths):
            for p in range(L):
                pool[tables[s][p // BS], g, p % BS] = dense_per_head[g][s][p]
    return pool


# ---------------------------------------------------------------------------
# hand-worked example
# ---------------------------------------------------------------------------
def test_golden_one_block(golden_dir):
    with open(os.path.join(golden_dir, "one_block_example.json")) as f:
        ex = json.load(f)
    d = ex["head_dim"]
    for placement in ex["placements"]:
        nb = placement["num_blocks"]
        blk = placement["table"][0]
        kp = np.full((nb, 1, BS, d), 100.0, dtype=np.float16)   # garbage elsewhere
        vp = np.full((nb, 1, BS, d), -100.0, dtype=np.float16)
        kp[blk, 0, :2] = _f16(ex["k"])
        vp[blk, 0, :2] = _f16(ex["v"])
        q = _f16(ex["q"]).reshape(1, 1, d)
        out = OA.paged_attention_decode(q, kp, vp, np.array([[blk]], np.int32),
                                        np.array([2], np.int32), ex["scale"], 1, "f16")
        np.testing.assert_allclose(out[0, 0], ex["expected_out"], rtol=0, atol=1e-13)
        np.testing.assert_allclose(out[0, 0], ex["expected_out_if_exact_ln3"], atol=1e-4)


# ---------------------------------------------------------------------------
# brute force on tiny inputs
# ---------------------------------------------------------------------------
def _brute_force(q_rows, dense_k, dense_v, lengths, scale, hq, hkv):
    """Per (s, h): explicit loops over tokens and dims, Python floats, math.exp."""
    group = hq // hkv
    out = []
    for s, L in enumerate(lengths):
        row = []
        for h in range(hq):
            g = h // group
            if L == 0:
                row.append([0.0] * len(q_rows[s][h]))
                continue
            logits = []
            for p in range(L):
                acc = 0.0
                for i in range(len(q_rows[s][h])):
                    acc += float(q_rows[s][h][i]) * float(dense_k[g][s][p][i])
                logits.append(scale * acc)
            top = max(logits)
            ws = [math.exp(z - top) for z in logits]
            tot = sum(ws)
            o = [0.0] * len(q_rows[s][h])
            for p in range(L):
                for i in range(len(o)):
                    o[i] += ws[p] / tot * float(dense_v[g][s][p][i])
            row.append(o)
        out.append(row)
    return np.array(out)


def _random_case(seed, lengths, hq, hkv, d, extra_blocks=3):
    rng = np.random.default_rng(seed)
    nbs = [-(-L // BS) for L in lengths]
    num_blocks = sum(nbs) + extra_blocks
    perm = rng.permutation(num_blocks)
    tables, pos = [], 0
    width = max(max(nbs), 1)
    for nb in nbs:
        tables.append(list(perm[pos:pos + nb]) + [-1] * (width - nb))
        pos += nb
    dense_k = [[rng.standard_normal((L, d)).astype(np.float16) for L in lengths] for _ in range(hkv)]
    dense_v = [[rng.standard_normal((L, d)).astype(np.float16) for L in lengths] for _ in range(hkv)]
    q = rng.standard_normal((len(lengths), hq, d)).astype(np.float16)
    kp = _pool_from_dense(dense_k, lengths, tables, num_blocks, d, fill=np.nan)
    vp = _pool_from_dense(dense_v, lengths, tables, num_blocks, d, fill=np.nan)
    return q, dense_k, dense_v, kp, vp, np.array(tables, np.int32), num_blocks


@pytest.mark.parametrize("seed,lengths,hq,hkv,d", [
    (0, [1, 5, 16, 17], 2, 2, 4),
    (1, [33, 2, 40], 4, 2, 8),       # GQA, 3 blocks, ragged tails
    (2, [48, 16, 31, 0], 6, 3, 4),   # exact multiples and an empty slot
    (3, [7], 8, 1, 2),               # MQA
])
def test_brute_force_tiny(seed, lengths, hq, hkv, d):
    q, dk, dv, kp, vp, tables, _ = _random_case(seed, lengths, hq, hkv, d)
    scale = 1.0 / math.sqrt(d)
    got = OA.paged_attention_decode(q, kp, vp, tables, np.array(lengths, np.int32), scale, hkv, "f16")
    want = _brute_force(q.astype(np.float64).tolist(), dk, dv, lengths, scale, hq, hkv)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms and special cases
# ---------------------------------------------------------------------------
def test_single_token_returns_v0_exactly():
    rng = np.random.default_rng(5)
    d = 8
    kp = rng.standard_normal((4, 1, BS, d)).astype(np.float16)
    vp = rng.standard_normal((4, 1, BS, d)).astype(np.float16)
    q = rng.standard_normal((1, 1, d)).astype(np.float16)
    out = OA.paged_attention_decode(q, kp, vp, np.array([[2]], np.int32), np.array([1], np.int32),
                                    0.3, 1, "f16")
    assert np.array_equal(out[0, 0], vp[2, 0, 0].astype(np.float64))


def test_equal_keys_and_zero_query_give_mean_of_v():
    rng = np.random.default_rng(6)
    d, L = 4, 37
    kp = rng.standard_normal((5, 1, BS, d)).astype(np.float16)
    vp = rng.standard_normal((5, 1, BS, d)).astype(np.float16)
    table = np.array([[4, 0, 3]], np.int32)
    dense_v = np.stack([vp[table[0, p // BS], 0, p % BS] for p in range(L)]).astype(np.float64)
    # q = 0: all logits are 0
    out = OA.paged_attention_decode(np.zeros((1, 1, d), np.float16), kp, vp, table,
                                    np.array([L], np.int32), 1.0, 1, "f16")
    np.testing.assert_allclose(out[0, 0], dense_v.mean(axis=0), rtol=0, atol=1e-14)
    # equal keys: every token's K is the same vector
    kp2 = kp.copy()
    kp2[:, 0] = kp[0, 0, 0]
    out2 = OA.paged_attention_decode(rng.standard_normal((1, 1, d)).astype(np.float16), kp2, vp,
                                     table, np.array([L], np.int32), 1.0, 1, "f16")
    np.testing.assert_allclose(out2[0, 0], dense_v.mean(axis=0), rtol=0, atol=1e-14)


def test_gqa_groups_read_their_own_kv_head():
    # V is the constant c_g on KV head g, so every query head of group g must output c_g.
    hq, hkv, d, L = 8, 4, 4, 20
    rng = np.random.default_rng(7)
    kp = rng.standard_normal((2, hkv, BS, d)).astype(np.float16)
    vp = np.zeros((2, hkv, BS, d), np.float16)
    consts = [1.5, -2.0, 0.25, 3.0]
    for g, c in enumerate(consts):
        vp[:, g] = c
    q = rng.standard_normal((1, hq, d)).astype(np.float16)
    out = OA.paged_attention_decode(q, kp, vp, np.array([[1, 0]], np.int32), np.array([L], np.int32),
                                    0.5, hkv, "f16")
    for h in range(hq):
        assert np.allclose(out[0, h], consts[h // (hq // hkv)], atol=1e-14)


def test_zero_length_sequence_outputs_zeros():
    q = np.ones((2, 1, 4), np.float16)
    kp = np.ones((2, 1, BS, 4), np.float16)
    out = OA.paged_attention_decode(q, kp, kp, np.array([[0], [-1]], np.int32),
                                    np.array([3, 0], np.int32), 1.0, 1, "f16")
    assert np.all(out[1] == 0.0) and np.all(np.isfinite(out[0]))


def test_bf16_conversion_exact():
    # 0x3F80 = 1.0, 0xC000 = -2.0, 0x7F7F = largest finite bf16, 0x0001 = smallest subnormal
    bits = np.array([0x3F80, 0xC000, 0x7F7F, 0x0001], np.uint16)
    got = to_f64(bits, "bf16")
    assert got[0] == 1.0 and got[1] == -2.0
    assert got[2] == (2 - 2 ** -7) * 2.0 ** 127
    assert got[3] == 2.0 ** -133
    assert round_to(np.array([1.0 + 2 ** -9]), "bf16")[0] == 1.0          # tie to even
    assert round_to(np.array([1.0 + 3 * 2 ** -9]), "bf16")[0] == 1.0 + 2 ** -7


# ---------------------------------------------------------------------------
# paging invariance: relabel physical blocks
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_permutation_of_physical_ids_leaves_output_unchanged(seed):
    lengths = [5, 17, 33, 64]
    q, _, _, kp, vp, tables, nb = _random_case(seed, lengths, 4, 4, 8, extra_blocks=10)
    lens = np.array(lengths, np.int32)
    base = OA.paged_attention_decode(q, kp, vp, tables, lens, 0.35, 4, "f16")
    pi = np.random.default_rng(100 + seed).permutation(nb)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[pi] = kp            # block b moves to pi[b]
    vp2[pi] = vp
    t2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1).astype(np.int32)
    moved = OA.paged_attention_decode(q, kp2, vp2, t2, lens, 0.35, 4, "f16")
    assert np.array_equal(base, moved)


# ---------------------------------------------------------------------------
# split-K closed form
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,P", [(1, 16), (100, 16), (100, 32), (513, 512), (2000, 512), (64, 64)])
def test_lse_merge_equals_unsplit_softmax(L, P):
    rng = np.random.default_rng(L + P)
    K = rng.standard_normal((L, 8)) * 3.0
    V = rng.standard_normal((L, 8))
    q = rng.standard_normal(8)
    whole = OA.attend(q, K, V, 0.9)
    merged = OA.lse_merge(OA.partition_partials(q, K, V, 0.9, P))
    np.testing.assert_allclose(merged, whole, rtol=1e-12, atol=1e-13)
    # one partition: the merge is the plain normalisation o / l
    m, l, o = OA.partition_partials(q, K, V, 0.9, max(L, 1))[0]
    np.testing.assert_allclose(o / l, whole, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# planted mistakes in a copy of the oracle must fail at least one pin
# ---------------------------------------------------------------------------
def _pins_pass(decode):
    """Run the brute-force, GQA and golden pins against a decode callable."""
    ok = True
    for seed, lengths, hq, hkv, d in [(1, [33, 2, 40], 4, 2, 8), (0, [1, 5, 16, 17], 2, 2, 4)]:
        q, dk, dv, kp, vp, tables, _ = _random_case(seed, lengths, hq, hkv, d)
        scale = 1.0 / math.sqrt(d)
        got = decode(q, kp, vp, tables, np.array(lengths, np.int32), scale, hkv)
        want = _brute_force(q.astype(np.float64).tolist(), dk, dv, lengths, scale, hq, hkv)
        ok &= bool(np.allclose(got, want, rtol=0, atol=1e-9, equal_nan=False))
    return ok


def _mutant_decode(kind):
    def decode(q, kp, vp, tables, lens, scale, hkv):
        qf, kf, vf = (to_f64(x, "f16") for x in (q, kp, vp))
        S, hq, d = qf.shape
        group = hq // hkv
        out = np.zeros((S, hq, d))
        for s in range(S):
            L = int(lens[s])
            for h in range(hq):
                g = (h % hkv) if kind == "gqa_modulo" else h // group
                if kind == "swap_block_slot":
                    idx = [(tables[s][p % BS] if p % BS < tables.shape[1] else 0, p // BS) for p in range(L)]
                else:
                    idx = [(tables[s][p // BS], p % BS) for p in range(L)]
                if kind == "off_by_one" and L > 1:
                    idx = idx[:-1]
                K = np.array([kf[b, g, o] for b, o in idx]).reshape(-1, d)
                V = np.array([vf[b, g, o] for b, o in idx]).reshape(-1, d)
                if kind == "swap_kv":
                    K, V = V, K
                sc = 1.0 if kind == "no_scale" else scale
                if K.shape[0] == 0:
                    continue
                z = sc * (K @ qf[s, h])
                e = np.exp(z - z.max())
                w = e if kind == "no_normalise" else e / e.sum()
                out[s, h] = w @ V
        return out
    return decode


def test_pins_accept_the_oracle():
    assert _pins_pass(lambda q, kp, vp, t, l, sc, hkv:
                      OA.paged_attention_decode(q, kp, vp, t, l, sc, hkv, "f16"))
    assert _pins_pass(_mutant_decode("none"))


@pytest.mark.parametrize("kind", ["gqa_modulo", "swap_block_slot", "off_by_one", "swap_kv",
                                  "no_scale", "no_normalise"])
def test_pins_reject_planted_mistakes(kind):
    with np.errstate(all="ignore"):
        try:
            passed = _pins_pass(_mutant_decode(kind))
        except (IndexError, ValueError):
            passed = False
    assert not passed, f"planted mistake {kind} slipped through the pins"
