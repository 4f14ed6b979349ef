"""Rounding of float64 values to the cache storage dtype.

The cache keeps rotated keys and values in its storage dtype ([Ch37]
"Keep layer, logical length, and capacity separate": fixed buffers
[B, H, C, d_h]; the pages use f64).  The oracle rounds each appended row once,
from its float64 value, with round-to-nearest-even, and keeps the rounded
value as a float64 number (every bf16 / f32 value is exactly a float64).

bfloat16 is written out from its definition: 1 sign bit, the 8-bit exponent
of binary32 (normal exponents -126 .. 127, subnormal spacing 2**-133) and a
7-bit fraction, so a value whose leading bit has exponent E >= -126 is rounded
to a multiple of 2**(E - 7), and smaller values to a multiple of 2**-133.
Magnitudes that round above the largest finite bf16 become infinities.
"""

import numpy as np

BF16_MAX = float.fromhex("0x1.fep127")  # (2 - 2**-7) * 2**127

DTYPES = ("bf16", "f32", "f64")


def round_to_bf16(x):
    """Nearest bfloat16 value (ties to even) of each float64 in ``x``, as float64."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    finite = np.isfinite(x)
    ax = np.abs(x[finite])
    _, e = np.frexp(ax)                      # ax = m * 2**e, m in [0.5, 1)
    lead = np.maximum(e - 1, -126)           # exponent of the leading bit, clamped to the subnormal range
    quantum = np.ldexp(1.0, lead - 7)        # spacing of bf16 numbers there
    r = np.rint(ax / quantum) * quantum      # division by a power of two is exact; rint ties to even
    r = np.where(r > BF16_MAX, np.inf, r)
    out[finite] = np.copysign(r, x[finite])
    return out


def round_to_f32(x):
    """Nearest binary32 value (ties to even) of each float64, as float64."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to(x, dtype):
    """Round float64 ``x`` to storage dtype ``dtype`` in {"bf16", "f32", "f64"}."""
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f32":
        return round_to_f32(x)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64).copy()
    raise ValueError(f"unknown storage dtype {dtype!r}")


def bf16_bits(x):
    """uint16 bit patterns of float64 values that are already bf16 numbers."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)
