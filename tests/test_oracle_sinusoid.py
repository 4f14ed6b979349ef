"""Pins of ``oracle.toy_decoder.sinusoidal_positions``, the additive positions of
the [LCP5] toy decoder (section "27 例得到的计算量与误差": sinusoidal absolute
positions, width 16).

The pins come from the mathematics of the sinusoid, not from its formula:

* PE(0) is (sin 0, cos 0) in every pair: exactly [0, 1, 0, 1, ...];
* within pair i, PE(p) is the unit vector (sin p w_i, cos p w_i), so moving from
  position p to p + k turns the pair by the angle k w_i: the pair's angle is
  read back with atan2 and compared with the frequency table of width 16,
  w_i = 10000^(-2i/16) = 10^(-i/2), written out as decimal numbers (1, 0.316...,
  0.1, ...);
* every pair has unit norm.
Planted mistakes -- sin and cos swapped, the exponent i/d instead of 2i/d, a
base of 1000 -- are run through the same checks and must fail them.
"""
import numpy as np
import pytest

from oracle.toy_decoder import sinusoidal_positions

D = 16
# 10^(-i/2) for i = 0 .. 7, as decimal literals
FREQ16 = np.array([1.0, 0.31622776601683794, 0.1, 0.031622776601683794, 0.01,
                   0.0031622776601683794, 0.001, 0.00031622776601683794])


def pin_failures(pe_fn):
    """Names of the pins that ``pe_fn(positions, d)`` fails (empty: all hold)."""
    bad = []
    pe0 = pe_fn([0], D)[0]
    if not np.array_equal(pe0, np.tile([0.0, 1.0], D // 2)):
        bad.append("PE(0)")
    p = np.arange(0, 2000, 7)
    pe = pe_fn(p, D)
    s, c = pe[:, 0::2], pe[:, 1::2]
    if np.abs(s * s + c * c - 1.0).max() > 1e-13:
        bad.append("unit pairs")
    # angle turned by one position step, per pair: atan2(sin, cos) of PE(1)
    pe1 = pe_fn([1], D)[0]
    w = np.arctan2(pe1[0::2], pe1[1::2])
    if np.abs(w - FREQ16).max() > 1e-15:
        bad.append("frequencies")
    # shift k: the pair turns by k w_i (compare as rotations, no retyped sinusoid)
    for k in (1, 5, 333):
        a = pe_fn(p, D)
        b = pe_fn(p + k, D)
        ang = k * FREQ16
        ca, sa = np.cos(ang), np.sin(ang)
        sb = a[:, 0::2] * ca + a[:, 1::2] * sa
        cb = a[:, 1::2] * ca - a[:, 0::2] * sa
        if max(np.abs(b[:, 0::2] - sb).max(), np.abs(b[:, 1::2] - cb).max()) > 1e-9:
            bad.append(f"shift {k}")
    return bad


def test_sinusoid_pins_hold():
    assert pin_failures(sinusoidal_positions) == []


def test_sinusoid_first_pair_is_sin_cos_of_the_position():
    pe = sinusoidal_positions([1, 2, 3], D)
    # sin 1, cos 1, sin 2, cos 2, sin 3, cos 3 to 12 digits (textbook values)
    want = [(0.841470984808, 0.540302305868), (0.909297426826, -0.416146836547),
            (0.141120008060, -0.989992496600)]
    assert np.abs(pe[:, :2] - np.array(want)).max() < 1e-12


def _swapped(positions, d):
    pe = sinusoidal_positions(positions, d)
    return pe[:, [i ^ 1 for i in range(d)]]


def _half_exponent(positions, d):
    pos = np.asarray(positions, dtype=np.float64)[:, None]
    i = np.arange(0, d, 2, dtype=np.float64)[None, :]
    ang = pos / np.power(10000.0, (i / 2) / d)
    out = np.zeros((pos.shape[0], d))
    out[:, 0::2], out[:, 1::2] = np.sin(ang), np.cos(ang)
    return out


def _base_1000(positions, d):
    pos = np.asarray(positions, dtype=np.float64)[:, None]
    i = np.arange(0, d, 2, dtype=np.float64)[None, :]
    ang = pos / np.power(1000.0, i / d)
    out = np.zeros((pos.shape[0], d))
    out[:, 0::2], out[:, 1::2] = np.sin(ang), np.cos(ang)
    return out


@pytest.mark.parametrize("planted", [_swapped, _half_exponent, _base_1000])
def test_planted_sinusoid_mistakes_fail_the_pins(planted):
    assert pin_failures(planted) != []
