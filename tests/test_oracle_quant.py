"""Pins of the INT8 KV-cache oracle: closed-form error bound, exact cases,
zero rows, code range, and decode over a cache whose values are exactly
representable (where it must equal the float decode)."""

import numpy as np
import pytest

from oracle import attention as OA
from oracle import quant as OQ
from oracle.block_manager import OracleBlockManager

BS = 16


def test_round_trip_error_is_at_most_half_a_step():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((500, 128)) * rng.uniform(0.01, 50, size=(500, 1))).astype(np.float32)
    c, s = OQ.quantize_rows(x)
    assert c.dtype == np.int8 and s.dtype == np.float32
    assert np.all(np.abs(c.astype(np.int32)) <= 127)
    err = np.abs(x.astype(np.float64) - OQ.dequantize(c, s))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-6))
    # the largest magnitude of each row maps to +-127
    assert np.all(np.abs(c).max(axis=1) == 127)


def test_exact_multiples_and_zero_rows():
    s = np.float32(0.25)
    codes = np.array([[-127, -3, 0, 5, 127], [1, 2, 3, 4, 127]], dtype=np.int32)
    x = (codes * s).astype(np.float32)
    c, sc = OQ.quantize_rows(x)
    assert np.all(sc == s) and np.array_equal(c.astype(np.int32), codes)
    z, zs = OQ.quantize_rows(np.zeros((2, 8), np.float32))
    assert np.all(z == 0) and np.all(zs == 0)
    # ties go to even: 2.5 steps -> 2, 3.5 -> 4
    xs = np.array([[2.5, 3.5, 127.0]], np.float32)
    c, sc = OQ.quantize_rows(xs)
    assert sc[0] == np.float32(1.0) and c.tolist() == [[2, 4, 127]]


def test_decode_over_exactly_representable_cache_equals_float_decode():
    rng = np.random.default_rng(1)
    nb, hkv, d = 10, 2, 8
    codes_k = rng.integers(-127, 128, size=(nb, hkv, BS, d)).astype(np.int8)
    codes_v = rng.integers(-127, 128, size=(nb, hkv, BS, d)).astype(np.int8)
    codes_k[..., 0] = 127                                   # max |c| = 127 in every row
    codes_v[..., 0] = -127
    sk = np.full((nb, hkv, BS), 2.0 ** -6, np.float32)
    sv = np.full((nb, hkv, BS), 2.0 ** -5, np.float32)
    kf = (codes_k.astype(np.float64) * 2.0 ** -6).astype(np.float16)   # exact in fp16
    vf = (codes_v.astype(np.float64) * 2.0 ** -5).astype(np.float16)
    q = rng.standard_normal((3, 4, d)).astype(np.float16)
    tables = np.array([[3, 1, 7], [0, 2, -1], [9, -1, -1]], np.int32)
    lens = np.array([40, 17, 5], np.int32)
    got = OQ.paged_attention_decode_int8(q, codes_k, codes_v, sk, sv, tables, lens, 0.4, hkv, "f16")
    want = OA.paged_attention_decode(q, kf, vf, tables, lens, 0.4, hkv, "f16")
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)
    # quantising those fp16 values gives back the same codes and scales
    c, s = OQ.quantize_rows(kf.astype(np.float32))
    assert np.array_equal(c, codes_k) and np.all(s == sk)


def test_quantised_write_lands_in_the_slots():
    bm = OracleBlockManager(6, initial_free_order=list(range(6)))
    bm.add_seq(0, 15)
    bm.add_seq(1, 16)
    slots = [bm.append_slot(0)[0], bm.append_slot(1)[0], -1]
    rng = np.random.default_rng(2)
    k = rng.standard_normal((3, 2, 8)).astype(np.float16)
    v = rng.standard_normal((3, 2, 8)).astype(np.float16)
    kc = np.zeros((6, 2, BS, 8), np.int8)
    ks = np.zeros((6, 2, BS), np.float32)
    nkc, nvc, nks, nvs = OQ.reshape_and_cache_int8(k, v, "f16", kc, kc, ks, ks, slots)
    for t in range(2):
        b, o = divmod(slots[t], BS)
        c, s = OQ.quantize_rows(k[t].astype(np.float32))
        assert np.array_equal(nkc[b, :, o], c) and np.array_equal(nks[b, :, o], s)
    written = {divmod(sl, BS) for sl in slots[:2]}
    for b in range(6):
        for o in range(BS):
            if (b, o) not in written:
                assert np.all(nkc[b, :, o] == 0) and np.all(nks[b, :, o] == 0)


@pytest.mark.parametrize("seed", [0, 1])
def test_int8_decode_error_vs_float_decode_is_small(seed):
    # a sanity bound, not a pin: quantisation error of N(0,1) data at d=64
    rng = np.random.default_rng(seed)
    nb, hkv, d = 8, 2, 64
    kf = rng.standard_normal((nb, hkv, BS, d)).astype(np.float16)
    vf = rng.standard_normal((nb, hkv, BS, d)).astype(np.float16)
    kc, ks = OQ.quantize_rows(kf.astype(np.float32))
    vc, vs = OQ.quantize_rows(vf.astype(np.float32))
    q = rng.standard_normal((2, 2, d)).astype(np.float16)
    tables = np.array([[0, 1, 2, 3], [4, 5, 6, 7]], np.int32)
    lens = np.array([64, 50], np.int32)
    a = OQ.paged_attention_decode_int8(q, kc, vc, ks, vs, tables, lens, d ** -0.5, hkv, "f16")
    b = OA.paged_attention_decode(q, kf, vf, tables, lens, d ** -0.5, hkv, "f16")
    assert np.abs(a - b).max() < 0.03
