"""Exact widening of cache values to float64 (oracle; test infrastructure only).

A bf16 value is the upper 16 bits of an IEEE float32, so placing its bit
pattern in the high half of a 32-bit word gives the float32 with the same
value, and float32 -> float64 is exact.  No rounding happens anywhere here.
"""

import numpy as np

DTYPES = ("f32", "bf16")


def widen(values, dtype):
    """Return ``values`` (float32 array, or uint16 bf16 bit patterns) as float64."""
    a = np.asarray(values)
    if dtype == "f32":
        if a.dtype != np.float32:
            raise TypeError("f32 data must be a float32 array")
        return a.astype(np.float64)
    if dtype == "bf16":
        if a.dtype != np.uint16:
            raise TypeError("bf16 data must be given as uint16 bit patterns")
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def bf16_bits_from_f64_exact(x):
    """bf16 bit patterns of values that are exactly representable in bf16.

    Used only to build special-case inputs (e.g. constant rows); raises if a
    value would need rounding, so no rounding rule is ever implied.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    if not np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64)):
        raise ValueError("value not exactly representable in float32")
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("value not exactly representable in bf16")
    return (u >> 16).astype(np.uint16)
