"""Exact conversions from the 16-bit storage types to float64.

Test infrastructure (see the package docstring).

The kernels store K, V, q and out as IEEE fp16 or bfloat16. NumPy has fp16
but no bfloat16, so bf16 arrays travel as their raw ``uint16`` bit patterns.
Both conversions below are exact: every fp16 and every bf16 value is
representable in float64.
"""

import numpy as np

F16 = "f16"
BF16 = "bf16"


def to_f64(arr, dtype):
    """Return ``arr`` (fp16 values, or bf16 bit patterns as uint16) as float64.

    bf16 is the upper half of an IEEE float32: shifting the 16 stored bits to
    the top of a 32-bit word gives the float32 with the same value.
    """
    a = np.asarray(arr)
    if dtype == F16:
        if a.dtype != np.float16:
            raise TypeError(f"fp16 data must be numpy float16, got {a.dtype}")
        return a.astype(np.float64)
    if dtype == BF16:
        if a.dtype != np.uint16:
            raise TypeError(f"bf16 data must be uint16 bit patterns, got {a.dtype}")
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def round_to(x, dtype):
    """Round float64 ``x`` to the storage type, nearest-even, and return float64.

    Used only to express "the oracle's value rounded to T" for the ulp
    diagnostic of the attention parity tests. fp16 uses NumPy's cast. bf16
    goes through float32 (exact for any value that later rounds to bf16
    except in double-rounding corner cases, which only affects the
    diagnostic, never a pass/fail bound) and then rounds the low 16 bits
    away with ties to even.
    """
    x = np.asarray(x, dtype=np.float64)
    if dtype == F16:
        return x.astype(np.float16).astype(np.float64)
    if dtype == BF16:
        u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
        lsb = (u >> 16) & 1
        r = ((u + 0x7FFF + lsb) >> 16) << 16
        return r.astype(np.uint32).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")
