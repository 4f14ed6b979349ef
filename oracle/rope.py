"""Rotary position embedding at absolute positions, float64.

[Ch37] section "Append along the position axis": the new key (and query) are
rotated for their absolute position, which is the zero-based old cache length;
the value is not rotated.  The pages print no frequency table or pairing, so
this module takes the RoFormer reading, stated once here:

* frequencies  theta_j = base ** (-2 j / d_h),  j = 0 .. d_h/2 - 1
* pairing      interleaved: features (2j, 2j+1) form pair j
* direction    (x, y) -> (x cos phi - y sin phi,  x sin phi + y cos phi),
               phi = p * theta_j.  Pinned by [Ch37] "Advance the layer cache
               one position at a time": head 1 at p = 1 stores
               (-0.841470985, 0.540302306) for the unit row (0, 1).

Angles are products p * theta_j in IEEE double; cos and sin come from the C
math library through Python's ``math`` module (one call per angle), so the
values do not depend on any vectorised trig implementation.  A base of 0 (or
None) switches the rotation off (identity), the configuration the [LCP5] toy
decoder needs, which uses additive sinusoidal positions instead.
"""

import math
from functools import lru_cache

import numpy as np


def inverse_frequencies(head_dim, base):
    """theta_j = base ** (-2 j / d_h) for j = 0 .. d_h/2 - 1, float64."""
    if head_dim <= 0 or head_dim % 2:
        raise ValueError(f"RoPE needs an even positive head width, got {head_dim}")
    return np.array([math.pow(base, -(2.0 * j) / head_dim) for j in range(head_dim // 2)],
                    dtype=np.float64)


@lru_cache(maxsize=64)
def _table(head_dim, base, max_position):
    inv = inverse_frequencies(head_dim, base)
    pos = np.arange(max_position + 1, dtype=np.float64)
    ang = pos[:, None] * inv[None, :]
    flat = ang.ravel()
    c = np.fromiter((math.cos(a) for a in flat), dtype=np.float64, count=flat.size)
    s = np.fromiter((math.sin(a) for a in flat), dtype=np.float64, count=flat.size)
    return c.reshape(ang.shape), s.reshape(ang.shape)


def cos_sin(positions, head_dim, base):
    """cos(phi), sin(phi) for phi = p * theta_j; shape positions.shape + (d_h/2,)."""
    pos = np.asarray(positions, dtype=np.int64)
    if pos.size and pos.min() < 0:
        raise ValueError("RoPE positions must be non-negative")
    top = int(pos.max()) if pos.size else 0
    c, s = _table(int(head_dim), float(base), top)
    return c[pos], s[pos]


def rotate(x, positions, base):
    """Rotate the last axis of ``x`` (float64, [..., d_h]) by its positions.

    ``positions`` broadcasts against ``x.shape[:-1]``.  Each product and each
    sum is one rounded float64 operation (NumPy does not fuse them).
    """
    x = np.asarray(x, dtype=np.float64)
    if not base:
        return x.copy()
    d = x.shape[-1]
    pos = np.broadcast_to(np.asarray(positions, dtype=np.int64), x.shape[:-1])
    c, s = cos_sin(pos, d, base)
    xe = x[..., 0::2]
    xo = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out
