"""Thin ctypes binding of libpaged_kv.so (the C ABI in include/paged_kv.h).

Argument marshalling only: tensor shapes become sizes, tensors become device
pointers, the current torch stream becomes the cudaStream_t. Every step of
the path runs in the library's CUDA kernels; there is no fallback. If the
library has not been built, every call raises ``LibraryNotBuilt``.

PyTorch supplies device memory and streams. The split-K workspace is a torch
allocation the binding keeps per (device, stream) and grows on demand.
"""

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpaged_kv.so")

STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
          3: "PKV_ERR_OUT_OF_BLOCKS", 4: "PKV_ERR_CUDA", 5: "PKV_ERR_WORKSPACE"}
PKV_F16, PKV_BF16 = 0, 1
BLOCK_SIZE = 16
NOALLOC_SCRATCH_BYTES = 32 << 20   # PKV_NOALLOC_SCRATCH_BYTES
BALANCED = -2                      # pkv_paged_attention_partition: balanced persistent schedule
SHARED_PREFIX = -5                 # pkv_paged_attention_partition: shared-prefix schedule

DEV_FLAGS = {0x1: "BAD_BLOCK_ID", 0x2: "BAD_CONTEXT_LEN", 0x4: "BAD_SLOT", 0x8: "BAD_PAIR",
             0x10: "WAIT_TIMEOUT", 0x20: "BAD_PLAN"}


class LibraryNotBuilt(RuntimeError):
    pass


class PagedKVError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        self.status_name = STATUS.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


class OutOfBlocks(PagedKVError):
    pass


_lib = None
_lib_lock = threading.Lock()

_c_int, _c_i64, _c_sz, _c_f, _c_p = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
_SIGS = {
    "pkv_version": ([], ctypes.c_char_p),
    "pkv_last_error_string": ([], ctypes.c_char_p),
    "pkv_device_status": ([ctypes.POINTER(ctypes.c_uint32), _c_int], _c_int),
    "pkv_paged_attention_decode": ([_c_p] * 6 + [_c_int] * 6 + [_c_f, _c_int, _c_int, _c_p, _c_sz, _c_p],
                                   _c_int),
    "pkv_paged_attention_decode_noalloc": ([_c_p] * 6 + [_c_int] * 6 + [_c_f, _c_int, _c_int, _c_p], _c_int),
    "pkv_paged_attention_decode_planned": ([_c_p] * 6 + [_c_int] * 6 + [_c_f, _c_int, _c_int, _c_p, _c_sz, _c_p],
                                           _c_int),
    "pkv_paged_attention_plan": ([_c_p, _c_p] + [_c_int] * 6 + [_c_p, _c_sz, _c_p], _c_int),
    "pkv_paged_attention_workspace_size": ([_c_int] * 6, _c_sz),
    "pkv_paged_attention_decode_sliding": ([_c_p] * 6 + [_c_int] * 6 + [_c_f, _c_int, _c_int, _c_int, _c_p, _c_sz,
                                                                       _c_p], _c_int),
    "pkv_paged_attention_sliding_workspace_size": ([_c_int] * 7, _c_sz),
    "pkv_paged_attention_partition": ([_c_int] * 6, _c_int),
    "pkv_reshape_and_cache": ([_c_p] * 5 + [_c_int] * 5 + [_c_p], _c_int),
    "pkv_copy_blocks": ([_c_p] * 3 + [_c_int] * 5 + [_c_p], _c_int),
    "pkv_check_copy_pairs": ([_c_p, _c_int, _c_int], _c_int),
    "pkv_reshape_and_cache_int8": ([_c_p, _c_p, _c_int] + [_c_p] * 5 + [_c_int] * 4 + [_c_p], _c_int),
    "pkv_paged_attention_decode_int8": ([_c_p] * 8 + [_c_int] * 6 + [_c_f, _c_int, _c_int, _c_p, _c_sz, _c_p],
                                        _c_int),
    "pkv_paged_attention_decode_int8_planned": ([_c_p] * 8 + [_c_int] * 6 + [_c_f, _c_int, _c_int, _c_p, _c_sz,
                                                                            _c_p], _c_int),
    "pkv_copy_blocks_int8": ([_c_p] * 5 + [_c_int] * 4 + [_c_p], _c_int),
    "pkv_selftest_bounded_wait": ([ctypes.c_uint32, _c_p], _c_int),
    "pkv_trace_enabled": ([], _c_int),
    "pkv_set_trace_buffer": ([_c_p, _c_int], _c_int),
    "pkv_trace_stamp": ([_c_p, _c_p], _c_int),
    "pkv_trace_empty_grid": ([_c_int, _c_int, _c_int, _c_p], _c_int),
    "pkv_bm_create": ([_c_int, _c_int, _c_p, ctypes.POINTER(_c_p)], _c_int),
    "pkv_bm_destroy": ([_c_p], None),
    "pkv_bm_add_seq": ([_c_p, _c_i64, _c_i64], _c_int),
    "pkv_bm_fork": ([_c_p, _c_i64, _c_i64], _c_int),
    "pkv_bm_append_slot": ([_c_p, _c_i64, _c_p, _c_p, _c_p], _c_int),
    "pkv_bm_append_slots": ([_c_p, _c_p, _c_int, _c_p, _c_p, _c_p], _c_int),
    "pkv_bm_free_seq": ([_c_p, _c_i64], _c_int),
    "pkv_bm_release_before": ([_c_p, _c_i64, _c_i64, _c_p], _c_int),
    "pkv_bm_beam_reorder": ([_c_p, _c_p, _c_int, _c_p, _c_p, _c_int], _c_int),
    "pkv_bm_add_seq_with_prefix": ([_c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_p], _c_int),
    "pkv_bm_block_tables": ([_c_p, _c_p, _c_int, _c_int, _c_p, _c_p], _c_int),
    "pkv_bm_refcount": ([_c_p, _c_int, _c_p], _c_int),
    "pkv_bm_seq_len": ([_c_p, _c_i64, _c_p], _c_int),
    "pkv_bm_num_free": ([_c_p], _c_int),
    "pkv_bm_num_seqs": ([_c_p], _c_int),
    "pkv_bm_free_stack": ([_c_p, _c_p, _c_int], _c_int),
}


def lib():
    """The loaded library (loaded on first use)."""
    global _lib
    if _lib is None:
        with _lib_lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise LibraryNotBuilt(
                        f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_217_gb300.build` "
                        "(nvcc, sm_103a); there is no CPU fallback")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (args, res) in _SIGS.items():
                    fn = getattr(handle, name)
                    fn.argtypes = args
                    fn.restype = res
                _lib = handle
    return _lib


def declared_symbols():
    return sorted(_SIGS)


def _check(status, what):
    if status != 0:
        msg = lib().pkv_last_error_string().decode(errors="replace")
        cls = OutOfBlocks if status == 3 else PagedKVError
        raise cls(status, f"{what}: {msg}")


def version():
    return lib().pkv_version().decode()


# ---------------------------------------------------------------------------
# device calls (torch tensors)
# ---------------------------------------------------------------------------
def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return PKV_F16
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (fp16 or bf16)")


def _need_cuda(*tensors):
    for t in tensors:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    dev = tensors[0].device
    if any(t.device != dev for t in tensors):
        raise ValueError("tensors must be on one device")


def _stream_ptr(device):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _launch(device, what, fn, *args):
    """Calls a launching entry point with ``device`` current and its current
    torch stream as the trailing cudaStream_t: the library looks up per-device
    state (the status word, the no-alloc scratch) on the current device, which
    must be the device of the tensors and of the stream."""
    import torch
    with torch.cuda.device(device):
        _check(fn(*args, _stream_ptr(device)), what)


_workspaces = {}


def _workspace(device, nbytes):
    import torch
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                   partition_size=0):
    return int(lib().pkv_paged_attention_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                         max_blocks_per_seq, partition_size))


def resolved_partition(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, partition_size=0):
    """Schedule a call runs with: BALANCED (-2), -1 (one pass per sequence and KV
    head) or the split-K partition size in tokens; 0 for invalid arguments."""
    return int(lib().pkv_paged_attention_partition(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                   max_blocks_per_seq, partition_size))


def paged_attention_decode(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                           num_kv_heads=None, partition_size=0, workspace=None, planned=False):
    """out[s, h] = softmax(scale * K_s q[s, h]) V_s over the paged cache (in place in ``out``).

    q, out: [S, Hq, D]; k_pool, v_pool: [num_blocks, Hkv, 16, D]; block_tables:
    int32 [S, max_blocks]; context_lens: int32 [S]. ``workspace`` (uint8 CUDA
    tensor) overrides the binding's own workspace. ``planned`` runs
    pkv_paged_attention_decode_planned, which uses the launch plan that
    paged_attention_plan left in the same workspace.
    """
    import torch
    _need_cuda(out, q, k_pool, v_pool, block_tables, context_lens)
    dt = _dtype_code(q)
    if out.dtype != q.dtype or k_pool.dtype != q.dtype or v_pool.dtype != q.dtype:
        raise TypeError("q, out, k_pool and v_pool must share one dtype")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    S, Hq, D = q.shape
    nb, hkv, bs, d2 = k_pool.shape
    if num_kv_heads is None:
        num_kv_heads = hkv
    if bs != BLOCK_SIZE or d2 != D or hkv != num_kv_heads or v_pool.shape != k_pool.shape:
        raise ValueError("pools must be [num_blocks, num_kv_heads, 16, head_dim]")
    if tuple(out.shape) != (S, Hq, D) or block_tables.dim() != 2 or block_tables.shape[0] != S \
            or tuple(context_lens.shape) != (S,):
        raise ValueError("shape mismatch among out, q, block_tables and context_lens")
    mb = block_tables.shape[1]
    need = workspace_size(S, Hq, num_kv_heads, D, mb, partition_size)
    ws_ptr, ws_bytes = None, 0
    if need:
        ws = workspace if workspace is not None else _workspace(q.device, need)
        ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    fn = lib().pkv_paged_attention_decode_planned if planned else lib().pkv_paged_attention_decode
    _launch(q.device, "paged_attention_decode_planned" if planned else "paged_attention_decode", fn,
            out.data_ptr(), q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), block_tables.data_ptr(),
            context_lens.data_ptr(), S, Hq, num_kv_heads, D, mb, nb, float(scale), dt, int(partition_size),
            ws_ptr, ws_bytes)
    return out


def paged_attention_plan(context_lens, block_tables, num_q_heads, num_kv_heads, head_dim, partition_size=0,
                         workspace=None):
    """The decode step's launch plan (pkv_paged_attention_plan) into ``workspace``
    (default: the binding's own workspace of the current stream, which
    paged_attention_decode(planned=True) then reads). block_tables: int32
    [S, max_blocks] (read by the shared-prefix schedule's plan)."""
    import torch
    _need_cuda(context_lens, block_tables)
    if context_lens.dtype != torch.int32 or context_lens.dim() != 1 or block_tables.dtype != torch.int32 \
            or block_tables.dim() != 2 or block_tables.shape[0] != context_lens.shape[0]:
        raise TypeError("context_lens must be int32 [S], block_tables int32 [S, max_blocks]")
    S, mb = block_tables.shape
    need = workspace_size(S, num_q_heads, num_kv_heads, head_dim, mb, partition_size)
    ws_ptr, ws_bytes = None, 0
    if need:
        ws = workspace if workspace is not None else _workspace(context_lens.device, need)
        ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    _launch(context_lens.device, "paged_attention_plan", lib().pkv_paged_attention_plan,
            context_lens.data_ptr(), block_tables.data_ptr(), S, int(num_q_heads), int(num_kv_heads),
            int(head_dim), int(mb), int(partition_size), ws_ptr, ws_bytes)


def sliding_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, sliding_window,
                           partition_size=0):
    return int(lib().pkv_paged_attention_sliding_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                                max_blocks_per_seq, sliding_window, partition_size))


def paged_attention_decode_sliding(out, q, k_pool, v_pool, block_tables, context_lens, scale, sliding_window,
                                   partition_size=0, workspace=None):
    """paged_attention_decode over each sequence's last ``sliding_window`` tokens
    (positions max(0, L - W) .. L-1); table entries before them are never read."""
    import torch
    _need_cuda(out, q, k_pool, v_pool, block_tables, context_lens)
    dt = _dtype_code(q)
    if out.dtype != q.dtype or k_pool.dtype != q.dtype or v_pool.dtype != q.dtype:
        raise TypeError("q, out, k_pool and v_pool must share one dtype")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    S, Hq, D = q.shape
    nb, hkv = k_pool.shape[0], k_pool.shape[1]
    if k_pool.shape[2:] != (BLOCK_SIZE, D) or v_pool.shape != k_pool.shape:
        raise ValueError("pools must be [num_blocks, num_kv_heads, 16, head_dim]")
    if tuple(out.shape) != (S, Hq, D) or block_tables.dim() != 2 or block_tables.shape[0] != S \
            or tuple(context_lens.shape) != (S,):
        raise ValueError("shape mismatch among out, q, block_tables and context_lens")
    mb = block_tables.shape[1]
    need = sliding_workspace_size(S, Hq, hkv, D, mb, int(sliding_window), partition_size)
    ws_ptr, ws_bytes = None, 0
    if need:
        ws = workspace if workspace is not None else _workspace(q.device, need)
        ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    _launch(q.device, "paged_attention_decode_sliding", lib().pkv_paged_attention_decode_sliding,
            out.data_ptr(), q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), block_tables.data_ptr(),
            context_lens.data_ptr(), S, Hq, hkv, D, mb, nb, float(scale), dt, int(sliding_window),
            int(partition_size), ws_ptr, ws_bytes)
    return out


def paged_attention_decode_noalloc(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                                   num_kv_heads=None, partition_size=0):
    """paged_attention_decode for callers that cannot allocate device memory.

    Split-K scratch comes from the library's fixed 32 MiB array instead of a
    workspace; see pkv_paged_attention_decode_noalloc in include/paged_kv.h
    (calls overlapping on the GPU race on that array).
    """
    import torch
    _need_cuda(out, q, k_pool, v_pool, block_tables, context_lens)
    dt = _dtype_code(q)
    if out.dtype != q.dtype or k_pool.dtype != q.dtype or v_pool.dtype != q.dtype:
        raise TypeError("q, out, k_pool and v_pool must share one dtype")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    S, Hq, D = q.shape
    nb, hkv = k_pool.shape[0], k_pool.shape[1]
    if num_kv_heads is None:
        num_kv_heads = hkv
    if k_pool.shape[2:] != (BLOCK_SIZE, D) or v_pool.shape != k_pool.shape or hkv != num_kv_heads:
        raise ValueError("pools must be [num_blocks, num_kv_heads, 16, head_dim]")
    if tuple(out.shape) != (S, Hq, D) or block_tables.dim() != 2 or block_tables.shape[0] != S \
            or tuple(context_lens.shape) != (S,):
        raise ValueError("shape mismatch among out, q, block_tables and context_lens")
    _launch(q.device, "paged_attention_decode_noalloc", lib().pkv_paged_attention_decode_noalloc,
            out.data_ptr(), q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), block_tables.data_ptr(),
            context_lens.data_ptr(), S, Hq, num_kv_heads, D, block_tables.shape[1], nb, float(scale), dt,
            int(partition_size))
    return out


def reshape_and_cache(k, v, k_pool, v_pool, slot_mapping):
    """k_pool[slot // 16, :, slot % 16] = k[t] (and v) for every token t with slot >= 0."""
    import torch
    _need_cuda(k, v, k_pool, v_pool, slot_mapping)
    dt = _dtype_code(k)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    T, hkv, D = k.shape
    if v.shape != k.shape or k_pool.shape[1:] != (hkv, BLOCK_SIZE, D) or v_pool.shape != k_pool.shape \
            or tuple(slot_mapping.shape) != (T,):
        raise ValueError("k, v: [T, Hkv, D]; pools: [num_blocks, Hkv, 16, D]; slot_mapping: [T]")
    if any(x.dtype != k.dtype for x in (v, k_pool, v_pool)):
        raise TypeError("k, v and pools must share one dtype")
    _launch(k.device, "reshape_and_cache", lib().pkv_reshape_and_cache,
            k.data_ptr(), v.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
            slot_mapping.data_ptr(), T, hkv, D, k_pool.shape[0], dt)


def copy_blocks(k_pool, v_pool, src_dst_pairs):
    """Copy block src to block dst in both pools for every row of src_dst_pairs (int64 [n, 2])."""
    import torch
    _need_cuda(k_pool, v_pool, src_dst_pairs)
    dt = _dtype_code(k_pool)
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be int64 [n, 2]")
    nb, hkv, bs, D = k_pool.shape
    _launch(k_pool.device, "copy_blocks", lib().pkv_copy_blocks,
            k_pool.data_ptr(), v_pool.data_ptr(), src_dst_pairs.data_ptr(),
            src_dst_pairs.shape[0], hkv, D, nb, dt)


# ---------------------------------------------------------------------------
# INT8 KV cache: int8 codes [num_blocks, Hkv, 16, D], fp32 scales [num_blocks, Hkv, 16]
# ---------------------------------------------------------------------------
def _check_int8_cache(k_cache, v_cache, k_scale, v_scale):
    import torch
    if k_cache.dtype != torch.int8 or v_cache.dtype != torch.int8:
        raise TypeError("k_cache and v_cache must be int8")
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32:
        raise TypeError("k_scale and v_scale must be float32")
    if k_cache.dim() != 4 or k_cache.shape[2] != BLOCK_SIZE or v_cache.shape != k_cache.shape \
            or tuple(k_scale.shape) != tuple(k_cache.shape[:3]) or v_scale.shape != k_scale.shape:
        raise ValueError("caches must be [num_blocks, Hkv, 16, D] and scales [num_blocks, Hkv, 16]")


def reshape_and_cache_int8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping):
    """Quantise each new K/V row (s = max|x|/127, c = rint(x/s)) into its slot of the INT8 cache."""
    import torch
    _need_cuda(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping)
    dt = _dtype_code(k)
    _check_int8_cache(k_cache, v_cache, k_scale, v_scale)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    T, hkv, D = k.shape
    if v.shape != k.shape or v.dtype != k.dtype or k_cache.shape[1:] != (hkv, BLOCK_SIZE, D) \
            or tuple(slot_mapping.shape) != (T,):
        raise ValueError("k, v: [T, Hkv, D]; caches: [num_blocks, Hkv, 16, D]; slot_mapping: [T]")
    _launch(k.device, "reshape_and_cache_int8", lib().pkv_reshape_and_cache_int8,
            k.data_ptr(), v.data_ptr(), dt, k_cache.data_ptr(), v_cache.data_ptr(), k_scale.data_ptr(),
            v_scale.data_ptr(), slot_mapping.data_ptr(), T, hkv, D, k_cache.shape[0])


def paged_attention_decode_int8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
                                partition_size=0, workspace=None, planned=False):
    """paged_attention_decode over the INT8 cache (K = c_K * s_K, V = c_V * s_V per row). ``planned``
    runs pkv_paged_attention_decode_int8_planned with the plan paged_attention_plan left in the same
    workspace."""
    import torch
    _need_cuda(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens)
    dt = _dtype_code(q)
    _check_int8_cache(k_cache, v_cache, k_scale, v_scale)
    if out.dtype != q.dtype:
        raise TypeError("q and out must share one dtype")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    S, Hq, D = q.shape
    nb, hkv = k_cache.shape[0], k_cache.shape[1]
    if k_cache.shape[3] != D or tuple(out.shape) != (S, Hq, D) or block_tables.dim() != 2 \
            or block_tables.shape[0] != S or tuple(context_lens.shape) != (S,):
        raise ValueError("shape mismatch among out, q, caches, block_tables and context_lens")
    mb = block_tables.shape[1]
    need = workspace_size(S, Hq, hkv, D, mb, partition_size)
    ws_ptr, ws_bytes = None, 0
    if need:
        ws = workspace if workspace is not None else _workspace(q.device, need)
        ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    fn = lib().pkv_paged_attention_decode_int8_planned if planned else lib().pkv_paged_attention_decode_int8
    _launch(q.device, "paged_attention_decode_int8_planned" if planned else "paged_attention_decode_int8", fn,
            out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), k_scale.data_ptr(),
            v_scale.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(), S, Hq, hkv, D, mb, nb,
            float(scale), dt, int(partition_size), ws_ptr, ws_bytes)
    return out


def copy_blocks_int8(k_cache, v_cache, k_scale, v_scale, src_dst_pairs):
    """copy_blocks for the INT8 cache: codes and scales of block src go to block dst."""
    import torch
    _need_cuda(k_cache, v_cache, k_scale, v_scale, src_dst_pairs)
    _check_int8_cache(k_cache, v_cache, k_scale, v_scale)
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be int64 [n, 2]")
    nb, hkv, _, D = k_cache.shape
    _launch(k_cache.device, "copy_blocks_int8", lib().pkv_copy_blocks_int8,
            k_cache.data_ptr(), v_cache.data_ptr(), k_scale.data_ptr(),
            v_scale.data_ptr(), src_dst_pairs.data_ptr(), src_dst_pairs.shape[0],
            hkv, D, nb)


def check_copy_pairs(pairs, num_blocks):
    """Host check: ids in range, distinct dst, no dst used as a src. Raises PagedKVError."""
    arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    _check(lib().pkv_check_copy_pairs(arr.ctypes.data, arr.shape[0], int(num_blocks)), "check_copy_pairs")


def device_status(clear=True):
    """Flags raised by the kernels' device-side index checks on the current device."""
    v = ctypes.c_uint32(0)
    _check(lib().pkv_device_status(ctypes.byref(v), 1 if clear else 0), "device_status")
    return int(v.value)


def selftest_bounded_wait(limit_us=2000):
    """Runs the bounded-wait self-test on the current device and stream (a wait
    that must run out and raise PKV_DEV_WAIT_TIMEOUT); read it with device_status()."""
    import torch
    _check(lib().pkv_selftest_bounded_wait(int(limit_us), _stream_ptr(torch.device("cuda", torch.cuda.current_device()))),
           "selftest_bounded_wait")


def trace_enabled():
    """True when the loaded library was built with per-CTA tracing (PKV_TRACE=1)."""
    return bool(lib().pkv_trace_enabled())


def set_trace_buffer(buffer):
    """Per-CTA phase timestamps of the following decode calls go into ``buffer``
    (an int64 CUDA tensor of 8 * records words), or stop with None."""
    if buffer is None:
        _check(lib().pkv_set_trace_buffer(None, 0), "set_trace_buffer")
        return
    _need_cuda(buffer)
    import torch
    if buffer.dtype != torch.int64 or buffer.numel() % 8:
        raise ValueError("the trace buffer is int64 with 8 words a record")
    _check(lib().pkv_set_trace_buffer(buffer.data_ptr(), buffer.numel() // 8), "set_trace_buffer")


def trace_stamp(words, index):
    """Enqueues on the current stream a write of the GPU clock (%globaltimer,
    ns) into ``words[index]`` (an int64 CUDA tensor) when the stream gets there."""
    _need_cuda(words)
    import torch
    if words.dtype != torch.int64 or not 0 <= index < words.numel() or not words.is_contiguous():
        raise ValueError("trace_stamp takes a contiguous int64 tensor and an index into it")
    ptr = words.data_ptr() + 8 * int(index)
    _launch(words.device, "trace_stamp", lib().pkv_trace_stamp, ptr)


def trace_empty_grid(device, ctas, threads, smem_bytes):
    """Enqueues on ``device``'s current stream a kernel of ``ctas`` CTAs x
    ``threads`` threads with ``smem_bytes`` of dynamic shared memory that does
    nothing, launched as the decode kernels are: timed between two events it
    is the fixed cost of a launch of that shape."""
    import torch
    device = torch.device(device)
    if device.type != "cuda":
        raise ValueError("trace_empty_grid needs a CUDA device")
    _launch(device, "trace_empty_grid", lib().pkv_trace_empty_grid, int(ctas), int(threads), int(smem_bytes))


def describe_device_flags(flags):
    return [name for bit, name in DEV_FLAGS.items() if flags & bit]


# ---------------------------------------------------------------------------
# host block manager
# ---------------------------------------------------------------------------
class BlockManager:
    """Host-side KV block manager (free stack, refcounts, copy-on-write).

    Wraps the library's C++ block manager; see pkv_bm_* in include/paged_kv.h.
    """

    def __init__(self, num_blocks, initial_free_order=None, block_size=BLOCK_SIZE):
        self._h = None
        self.num_blocks = int(num_blocks)
        order = None
        if initial_free_order is not None:
            order = np.ascontiguousarray(np.asarray(initial_free_order, dtype=np.int32))
            if order.shape != (self.num_blocks,):
                raise ValueError("initial_free_order must have num_blocks entries")
        h = ctypes.c_void_p()
        _check(lib().pkv_bm_create(self.num_blocks, int(block_size),
                                   None if order is None else order.ctypes.data, ctypes.byref(h)),
               "bm_create")
        self._h = h

    def close(self):
        if self._h is not None:
            lib().pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq_id, num_tokens):
        _check(lib().pkv_bm_add_seq(self._h, int(seq_id), int(num_tokens)), "bm_add_seq")

    def fork(self, parent, child):
        _check(lib().pkv_bm_fork(self._h, int(parent), int(child)), "bm_fork")

    def append_slot(self, seq_id):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib().pkv_bm_append_slot(self._h, int(seq_id), ctypes.byref(slot), ctypes.byref(src),
                                        ctypes.byref(dst)), "bm_append_slot")
        return slot.value, src.value, dst.value

    def append_slots(self, seq_ids):
        """One slot per sequence, in order; returns (slots int64 [n], pairs int64 [p, 2])."""
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ids.shape[0]
        slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        np_ = ctypes.c_int()
        _check(lib().pkv_bm_append_slots(self._h, ids.ctypes.data, n, slots.ctypes.data, pairs.ctypes.data,
                                         ctypes.byref(np_)), "bm_append_slots")
        return slots, pairs[:np_.value].copy()

    def free_seq(self, seq_id):
        _check(lib().pkv_bm_free_seq(self._h, int(seq_id)), "bm_free_seq")

    def beam_reorder(self, old_ids, parents, new_ids):
        """Beam step: new beam i continues old beam old_ids[parents[i]]; the old beams are dropped."""
        o = np.ascontiguousarray(np.asarray(old_ids, dtype=np.int64))
        p = np.ascontiguousarray(np.asarray(parents, dtype=np.int32))
        n = np.ascontiguousarray(np.asarray(new_ids, dtype=np.int64))
        _check(lib().pkv_bm_beam_reorder(self._h, o.ctypes.data, o.shape[0], p.ctypes.data, n.ctypes.data,
                                         n.shape[0]), "bm_beam_reorder")

    def add_seq_with_prefix(self, seq_id, num_tokens, donor, prefix_tokens):
        """New sequence sharing the whole blocks of its common prefix with `donor`;
        returns the number of shared positions (a multiple of 16)."""
        out = ctypes.c_int64()
        _check(lib().pkv_bm_add_seq_with_prefix(self._h, int(seq_id), int(num_tokens), int(donor),
                                                int(prefix_tokens), ctypes.byref(out)), "bm_add_seq_with_prefix")
        return out.value

    def release_before(self, seq_id, first_token):
        """Drops the sequence's hold on blocks wholly before position first_token
        (their table entries become -1); returns how many entries were dropped."""
        n = ctypes.c_int()
        _check(lib().pkv_bm_release_before(self._h, int(seq_id), int(first_token), ctypes.byref(n)),
               "bm_release_before")
        return n.value

    def block_tables(self, seq_ids, max_blocks_per_seq):
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ids.shape[0]
        table = np.empty((n, int(max_blocks_per_seq)), dtype=np.int32)
        lens = np.empty(n, dtype=np.int32)
        _check(lib().pkv_bm_block_tables(self._h, ids.ctypes.data, n, int(max_blocks_per_seq),
                                         table.ctypes.data, lens.ctypes.data), "bm_block_tables")
        return table, lens

    def block_table(self, seq_id):
        n = -(-self.seq_len(seq_id) // BLOCK_SIZE)
        t, _ = self.block_tables([seq_id], max(n, 1))
        return t[0, :n].tolist()

    def refcount(self, block):
        out = ctypes.c_int32()
        _check(lib().pkv_bm_refcount(self._h, int(block), ctypes.byref(out)), "bm_refcount")
        return out.value

    def seq_len(self, seq_id):
        out = ctypes.c_int64()
        _check(lib().pkv_bm_seq_len(self._h, int(seq_id), ctypes.byref(out)), "bm_seq_len")
        return out.value

    def num_free(self):
        return int(lib().pkv_bm_num_free(self._h))

    def num_seqs(self):
        return int(lib().pkv_bm_num_seqs(self._h))

    def free_stack(self):
        n = int(lib().pkv_bm_free_stack(self._h, None, 0))
        out = np.empty(max(n, 1), dtype=np.int32)
        lib().pkv_bm_free_stack(self._h, out.ctypes.data, n)
        return out[:n].tolist()
