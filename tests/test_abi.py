"""The C-ABI library without a GPU: it loads, exports every function that
include/paged_kv.h declares, sizes workspaces, picks partitions, and rejects
bad arguments on the host before anything would be launched."""

import ctypes
import os
import re

import pytest

from paged_kv_cache_217_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        with open(os.path.join(ROOT, "include", fn)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_function():
    lib = B.lib()
    declared = _declared_functions()
    assert len(declared) >= 20
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert sorted(declared) == B.declared_symbols()
    assert B.version().startswith("paged_kv")


def _round16(x):
    return (x + 15) // 16 * 16


def _split_bytes(S, hq, hkv, d, parts):
    """Fixed partitions: fp32 partials [S][Hq][P][D], (max, sum) [S][Hq][P], counters [S][Hkv]."""
    return _round16(S * hq * parts * (d * 4 + 8) + S * hkv * 4)


def _balanced_bytes(S, hq, hkv, d):
    """Balanced schedule: two slots per persistent warp (2048 warps max), counters [S][Hkv]."""
    slot_floats = ((hq // hkv) * (d + 2) + 3) // 4 * 4
    return _round16(2 * 2048 * slot_floats * 4 + S * hkv * 4)


def _plan_bytes(S):
    """Launch plan: a 16-byte header, the order int32[S] (16-byte rounded), then
    int4[2 S] of rows {sequence, length, block ids 0..5}."""
    return 16 + _round16(4 * S) + 32 * S


def test_workspace_and_partition_choice():
    # automatic choice: one CTA per (sequence, KV head) with at least 608 pairs
    assert B.resolved_partition(64, 40, 40, 128, 32) == -1          # 2560 pairs
    assert B.resolved_partition(256, 32, 8, 128, 64) == -1          # 2048 pairs
    # 2..1024 sequences in a grid of at most 4096 CTAs: a launch plan region, a
    # 16-byte header, int32[num_seqs] (16-byte rounded) and two int4 rows a sequence
    assert B.workspace_size(64, 40, 40, 128, 32) == 16 + 256 + 64 * 32
    assert B.workspace_size(256, 32, 8, 128, 64) == 16 + 256 * 4 + 256 * 32
    assert B.workspace_size(130, 8, 8, 128, 64) == 16 + 528 + 130 * 32    # 130 * 4 rounded up to 16
    assert B.workspace_size(2, 8, 8, 128, 1) == _plan_bytes(2)
    assert B.workspace_size(1, 8, 8, 128, 1) == 0                    # one sequence: nothing to order
    assert B.workspace_size(512, 16, 16, 128, 64) == 0               # 8192 CTAs: no long-first order
    assert B.workspace_size(1025, 1, 1, 128, 64) == 0                # beyond the plan's 1024 sequences
    assert B.resolved_partition(8, 96, 96, 128, 2048) == -1         # 768 pairs
    # fewer pairs: partitions just large enough for 608 CTAs, at least 256 tokens
    assert B.resolved_partition(2, 8, 8, 128, 2048) == 864          # 16 pairs x 38 parts
    assert B.workspace_size(2, 8, 8, 128, 2048) == _split_bytes(2, 8, 8, 128, 38) + _plan_bytes(2)
    assert B.resolved_partition(4, 4, 4, 64, 100) == 256            # 16 pairs, 1600 tokens
    assert B.resolved_partition(4, 4, 4, 64, 16) == -1              # 256 tokens: one pass
    # the shared-prefix schedule, on request: two partial slots, then the
    # prefix plan (header, groups int4[S / 2], shared tokens int32[S])
    assert B.resolved_partition(128, 72, 72, 128, 80, B.SHARED_PREFIX) == B.SHARED_PREFIX
    assert B.workspace_size(128, 72, 72, 128, 80, B.SHARED_PREFIX) == \
        _split_bytes(128, 72, 72, 128, 4) + 16 + 64 * 16 + 128 * 16 + 512   # partials of 4 chunks, the plan
    assert B.resolved_partition(128, 64, 8, 128, 80, B.SHARED_PREFIX) == 0     # 8 query heads per KV head
    assert B.resolved_partition(1, 8, 8, 128, 80, B.SHARED_PREFIX) == 0        # one sequence
    assert B.resolved_partition(8, 8, 8, 128, 257, B.SHARED_PREFIX) == 0       # tables wider than 256 blocks
    # the balanced persistent schedule, on request
    assert B.resolved_partition(64, 40, 40, 128, 32, -2) == B.BALANCED
    assert B.workspace_size(64, 40, 40, 128, 32, -2) == _balanced_bytes(64, 40, 40, 128)
    assert B.workspace_size(256, 32, 8, 128, 64, -2) == _balanced_bytes(256, 32, 8, 128)
    # explicit choices
    assert B.resolved_partition(8, 96, 96, 128, 2048, -1) == -1
    assert B.resolved_partition(8, 96, 96, 128, 2048, 256) == 256
    assert B.workspace_size(8, 96, 96, 128, 2048, -1) == _plan_bytes(8)   # 768 CTAs: the plan region
    assert B.workspace_size(8, 96, 96, 128, 2048, 512) == _split_bytes(8, 96, 96, 128, 64)  # 49152 CTAs
    assert B.workspace_size(3, 6, 2, 64, 10, 16) == _split_bytes(3, 6, 2, 64, 10) + _plan_bytes(3)
    # a partition that covers the whole context is one pass
    assert B.resolved_partition(4, 4, 4, 64, 4, 64) == -1
    assert B.workspace_size(4, 4, 4, 64, 4, 64) == _plan_bytes(4)
    # invalid partition sizes
    assert B.resolved_partition(4, 4, 4, 64, 4, 24) == 0
    assert B.workspace_size(0, 4, 4, 64, 4) == 0


FAKE = 0x10000  # a 16-byte aligned address; never dereferenced because every call below fails its checks


def _decode(**kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, S=4, Hq=4, Hkv=4, D=64, MB=4, NB=64,
             scale=0.125, dt=B.PKV_F16, part=0, ws=None, wsb=0)
    a.update(kw)
    st = B.lib().pkv_paged_attention_decode(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["S"], a["Hq"],
                                            a["Hkv"], a["D"], a["MB"], a["NB"], a["scale"], a["dt"], a["part"],
                                            a["ws"], a["wsb"], None)
    return st, B.lib().pkv_last_error_string().decode()


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), 1),           # not a multiple
    (dict(Hq=32, Hkv=2), 2),          # group 16 > 8
    (dict(D=80), 2),                  # head_dim
    (dict(dt=7), 2),                  # dtype
    (dict(MB=0), 1),
    (dict(NB=0), 1),
    (dict(S=70000), 2),
    (dict(scale=float("inf")), 1),
    (dict(q=None), 1),
    (dict(q=FAKE + 8), 1),            # misaligned
    (dict(part=24), 1),               # not a multiple of 16
    (dict(MB=64, part=16), 5),        # split needs a workspace
    (dict(MB=64, part=16, ws=FAKE, wsb=100), 5),
    (dict(part=-2), 5),               # the balanced schedule needs one too
    (dict(part=-2, S=4000, MB=4), 2),  # beyond the balanced schedule's batch limit
])
def test_decode_rejects_bad_arguments_before_launch(kw, status):
    st, msg = _decode(**kw)
    assert st == status, msg
    assert msg


def test_zero_sequences_is_a_no_op():
    assert _decode(S=0, out=None, q=None)[0] == 0


def test_cache_ops_reject_bad_arguments():
    L = B.lib()
    assert L.pkv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 64, 8, 0, None) == 0   # no tokens
    assert L.pkv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 4, 64, 8, 0, None) == 1
    assert L.pkv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 60, 8, 0, None) == 2
    assert L.pkv_reshape_and_cache(FAKE + 4, FAKE, FAKE, FAKE, FAKE, 2, 4, 64, 8, 0, None) == 1
    assert L.pkv_reshape_and_cache(None, FAKE, FAKE, FAKE, FAKE, 2, 4, 64, 8, 0, None) == 1
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 0, 4, 64, 8, 0, None) == 0                     # no pairs
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, -1, 4, 64, 8, 0, None) == 1
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 70000, 4, 64, 8, 0, None) == 2
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE + 4, 2, 4, 64, 8, 0, None) == 1
    assert L.pkv_copy_blocks(FAKE, FAKE, FAKE, 2, 4, 64, 8, 9, None) == 2


def test_device_status_needs_an_argument():
    assert B.lib().pkv_device_status(None, 0) == 1


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", "/nonexistent/libpaged_kv.so")
    with pytest.raises(B.LibraryNotBuilt):
        B.lib()


def test_tracing_is_off_in_the_default_build():
    assert B.trace_enabled() is False
    assert B.lib().pkv_set_trace_buffer(None, 0) == 2          # PKV_ERR_UNSUPPORTED
    # the clock stamp exists in every build and checks its word on the host
    assert B.lib().pkv_trace_stamp(None, None) == 1             # PKV_ERR_INVALID_ARG
    assert B.lib().pkv_trace_stamp(ctypes.c_void_p(12), None) == 1
    # so does the empty grid (its shape is checked before any launch)
    for ctas, threads, smem in [(0, 96, 0), (1, 0, 0), (1, 1025, 0), (1, 32, -1), (1, 32, 227 * 1024 + 1)]:
        assert B.lib().pkv_trace_empty_grid(ctas, threads, smem, None) == 1, (ctas, threads, smem)


def test_binding_scratch_size_matches_the_header():
    # the binding restates PKV_NOALLOC_SCRATCH_BYTES; both must change together
    with open(os.path.join(ROOT, "include", "paged_kv.h")) as f:
        text = f.read()
    m = re.search(r"#define\s+PKV_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "PKV_NOALLOC_SCRATCH_BYTES not found in include/paged_kv.h"
    assert int(m.group(1)) << int(m.group(2)) == B.NOALLOC_SCRATCH_BYTES


def test_plan_rejects_bad_arguments_before_launch():
    plan = B.lib().pkv_paged_attention_plan
    assert plan(None, None, 4, 4, 4, 64, 4, 0, FAKE, 64, None) == 1          # no lengths
    assert plan(FAKE + 2, None, 4, 4, 4, 64, 4, 0, FAKE, 64, None) == 1      # misaligned lengths
    assert plan(FAKE, None, 4, 6, 4, 64, 4, 0, FAKE, 64, None) == 1          # not a multiple
    assert plan(FAKE, None, 4, 4, 4, 64, 4, 0, None, 0, None) == 5           # needs the plan region
    assert plan(FAKE, None, 4, 4, 4, 64, 4, 0, FAKE, 31, None) == 5          # 16 + 16 bytes
    assert plan(FAKE, None, 4, 4, 4, 64, 4, 24, FAKE, 64, None) == 1         # bad partition
    assert plan(FAKE, None, 0, 4, 4, 64, 4, 0, None, 0, None) == 0           # nothing to plan
    assert plan(FAKE, None, 1, 4, 4, 64, 4, 0, None, 0, None) == 0           # one sequence: nothing to plan
    # the shared-prefix plan reads the tables
    assert plan(FAKE, None, 4, 4, 4, 64, 4, -5, FAKE, 1 << 20, None) == 1
    assert plan(FAKE, FAKE, 4, 16, 2, 64, 4, -5, FAKE, 1 << 20, None) == 2   # 8 query heads per KV head
    assert plan(FAKE, FAKE, 4, 4, 4, 64, 300, -5, FAKE, 1 << 30, None) == 2  # tables wider than 256 blocks
    assert plan(FAKE, FAKE, 4, 4, 4, 64, 4, -5, FAKE, 64, None) == 5         # workspace too small
