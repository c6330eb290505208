"""GPU parity of reshape_and_cache and copy_blocks (through the C ABI): bit-exact
against the oracle copies, untouched bytes included."""

import numpy as np
import pytest
import torch

import helpers as H
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


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hkv,d", [(4, 64), (8, 128), (2, 256), (72, 128)])
def test_reshape_and_cache_bit_exact(dtype, hkv, d):
    nb, T = 40, 97
    rng = np.random.default_rng(hkv + d)
    slots = rng.choice(nb * 16, size=T, replace=False).astype(np.int64)
    slots[::7] = -1                                  # skipped tokens
    kp = W.normal_values((nb, hkv, 16, d), dtype, 1, "cuda")
    vp = W.normal_values((nb, hkv, 16, d), dtype, 2, "cuda")
    k = W.normal_values((T, hkv, d), dtype, 3, "cuda")
    v = W.normal_values((T, hkv, d), dtype, 4, "cuda")
    kb, vb = _bits(kp), _bits(vp)
    B.reshape_and_cache(k, v, kp, vp, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    ek, ev = OC.reshape_and_cache(_bits(k), _bits(v), kb, vb, slots)
    assert np.array_equal(_bits(kp), ek) and np.array_equal(_bits(vp), ev)
    assert B.device_status(clear=True) == 0


def test_reshape_llama3_8b_step_slots():
    # one new token per sequence of the Llama-3-8B-shaped batch, at its last position
    shape = W.llama3_8b_gqa_decode(0)
    lens = shape.context_lens
    nb = W.pool_size(lens)
    tables, _ = W.scattered_tables(lens, nb, 0)
    slots = np.array([tables[s, (L - 1) // 16] * 16 + (L - 1) % 16 for s, L in enumerate(lens.tolist())],
                     np.int64)
    kp = W.normal_values((nb, 8, 16, 128), "bf16", 1, "cuda")
    vp = W.normal_values((nb, 8, 16, 128), "bf16", 2, "cuda")
    k = W.normal_values((256, 8, 128), "bf16", 3, "cuda")
    v = W.normal_values((256, 8, 128), "bf16", 4, "cuda")
    kb, vb = _bits(kp), _bits(vp)
    B.reshape_and_cache(k, v, kp, vp, torch.from_numpy(slots).cuda())
    ek, ev = OC.reshape_and_cache(_bits(k), _bits(v), kb, vb, slots)
    assert np.array_equal(_bits(kp), ek) and np.array_equal(_bits(vp), ev)


def test_reshape_flags_slot_outside_pool():
    kp = W.normal_values((4, 2, 16, 64), "f16", 1, "cuda")
    vp = W.normal_values((4, 2, 16, 64), "f16", 2, "cuda")
    k = W.normal_values((2, 2, 64), "f16", 3, "cuda")
    kb = _bits(kp)
    B.device_status(clear=True)
    B.reshape_and_cache(k, k, kp, vp, torch.tensor([64, 3], dtype=torch.int64, device="cuda"))
    assert B.device_status(clear=True) & 0x4
    ek, _ = OC.reshape_and_cache(_bits(k)[1:], _bits(k)[1:], kb, kb, np.array([3]))
    assert np.array_equal(_bits(kp), ek)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hkv,d", [(4, 64), (72, 128), (3, 256)])
def test_copy_blocks_bit_exact(dtype, hkv, d):
    nb = 50
    rng = np.random.default_rng(d)
    ids = rng.permutation(nb)
    pairs = np.stack([ids[:12], ids[12:24]], axis=1).astype(np.int64)
    pairs[3, 0] = pairs[2, 0]                        # one source copied twice
    B.check_copy_pairs(pairs, nb)
    kp = W.normal_values((nb, hkv, 16, d), dtype, 5, "cuda")
    vp = W.normal_values((nb, hkv, 16, d), dtype, 6, "cuda")
    kb, vb = _bits(kp), _bits(vp)
    B.copy_blocks(kp, vp, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    ek, ev = OC.copy_blocks(kb, vb, pairs)
    assert np.array_equal(_bits(kp), ek) and np.array_equal(_bits(vp), ev)
    assert B.device_status(clear=True) == 0


def test_copy_blocks_flags_bad_pair_and_copies_the_rest():
    kp = W.normal_values((6, 2, 16, 64), "f16", 7, "cuda")
    vp = W.normal_values((6, 2, 16, 64), "f16", 8, "cuda")
    kb, vb = _bits(kp), _bits(vp)
    B.device_status(clear=True)
    B.copy_blocks(kp, vp, torch.tensor([[1, 2], [0, 9]], dtype=torch.int64, device="cuda"))
    assert B.device_status(clear=True) & 0x8
    ek, ev = OC.copy_blocks(kb, vb, np.array([[1, 2]]))
    assert np.array_equal(_bits(kp), ek) and np.array_equal(_bits(vp), ev)
