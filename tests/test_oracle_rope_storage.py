"""Pins of oracle.rope and oracle.storage against closed forms, a matrix
exponential, the [Ch37] printed rotation and torch's bf16 cast."""
import math

import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import rope, storage


def test_inverse_frequencies_closed_form():
    d, base = 128, 10000.0
    inv = rope.inverse_frequencies(d, base)
    assert inv[0] == 1.0
    ref = np.exp(-np.log(base) * (2.0 * np.arange(d // 2)) / d)
    np.testing.assert_allclose(inv, ref, rtol=4e-15, atol=0)
    assert np.all(np.diff(inv) < 0)


def test_two_dim_rotation_is_rotation_by_p_radians():
    # d_h = 2 has the single frequency theta_0 = 1: the rotation angle is p rad.
    for p in [0, 1, 2, 7, 100, 4095]:
        for x in [(1.0, 0.0), (0.0, 1.0), (0.3, -2.5)]:
            r = rope.rotate(np.array(x), p, 10000.0)
            c, s = math.cos(p), math.sin(p)
            assert r[0] == pytest.approx(x[0] * c - x[1] * s, abs=1e-15)
            assert r[1] == pytest.approx(x[0] * s + x[1] * c, abs=1e-15)


def test_page_rotation_direction():
    # [Ch37] "Advance the layer cache one position at a time": head 1 stores
    # (-0.841470985, 0.540302306) for (0, 1) at p = 1 and (-1.325444263, 0.493150590)
    # for (1, 1) at p = 2 (9 printed decimals).
    r1 = rope.rotate(np.array([0.0, 1.0]), 1, 10000.0)
    r2 = rope.rotate(np.array([1.0, 1.0]), 2, 10000.0)
    np.testing.assert_allclose(r1, [-0.841470985, 0.540302306], atol=6e-10)
    np.testing.assert_allclose(r2, [-1.325444263, 0.493150590], atol=6e-10)


@pytest.mark.parametrize("d", [4, 8, 16])
def test_block_rotation_matches_matrix_exponential(d):
    # RoPE is the flow of dx/dp = A x with A block-diagonal [[0,-t_j],[t_j,0]] on
    # interleaved pairs: R(p) = expm(p A).  Pins pairing, direction and frequencies.
    base = 10000.0
    theta = np.exp(-np.log(base) * (2.0 * np.arange(d // 2)) / d)
    A = np.zeros((d, d))
    for j, t in enumerate(theta):
        A[2 * j + 1, 2 * j] = t
        A[2 * j, 2 * j + 1] = -t
    rng = np.random.default_rng(1)
    x = rng.normal(size=d)
    for p in [0, 1, 3, 17, 40]:
        ref = scipy.linalg.expm(p * A) @ x
        np.testing.assert_allclose(rope.rotate(x, p, base), ref, atol=1e-11)


def test_rotation_preserves_norm_and_relative_scores():
    rng = np.random.default_rng(2)
    q = rng.normal(size=(5, 128))
    k = rng.normal(size=(5, 128))
    m = np.array([0, 3, 100, 900, 4000])
    n = np.array([0, 1, 50, 899, 10])
    qr, kr = rope.rotate(q, m, 10000.0), rope.rotate(k, n, 10000.0)
    np.testing.assert_allclose(np.linalg.norm(qr, axis=1), np.linalg.norm(q, axis=1), rtol=1e-13)
    # q(m) . k(n) depends on m - n only: shift both positions by the same amount.
    for shift in [1, 77, 10000]:
        qs, ks = rope.rotate(q, m + shift, 10000.0), rope.rotate(k, n + shift, 10000.0)
        np.testing.assert_allclose((qs * ks).sum(1), (qr * kr).sum(1), atol=1e-9)
    # ... and does change when only one side moves.
    qs = rope.rotate(q, m + 1, 10000.0)
    assert np.abs((qs * kr).sum(1) - (qr * kr).sum(1)).max() > 1e-3


def test_position_zero_and_rope_off_are_identity():
    x = np.random.default_rng(3).normal(size=(3, 64))
    np.testing.assert_array_equal(rope.rotate(x, 0, 10000.0), x)
    np.testing.assert_array_equal(rope.rotate(x, [5, 6, 7], 0), x)


def test_bf16_matches_torch_cast_for_binary32_inputs():
    rng = np.random.default_rng(4)
    vals = np.concatenate([
        rng.normal(size=200000).astype(np.float32),
        (rng.normal(size=20000) * 1e-38).astype(np.float32),    # binary32/bf16 subnormals
        np.clip(rng.normal(size=20000) * 3e38, -3.4e38, 3.4e38).astype(np.float32),  # top of the range
        np.array([0.0, -0.0, 1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 3.3895314e38, 3.40e38], np.float32),
    ]).astype(np.float32)
    mine = storage.round_to_bf16(vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(mine, ref)
    assert np.array_equal(np.signbit(mine), np.signbit(ref))


def _bf16_neighbours(r):
    bits = storage.bf16_bits(r).astype(np.uint32)
    up = ((bits + 1) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    dn = ((bits - 1) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    return dn, up


def test_bf16_is_nearest_with_ties_to_even_brute_force():
    # float64 values that are not binary32 numbers (so no cast can hide double rounding)
    rng = np.random.default_rng(5)
    x = rng.normal(size=100000) * np.exp2(rng.integers(-20, 20, 100000))
    x = x + np.exp2(np.floor(np.log2(np.abs(x))) - 40)  # bits below binary32 precision
    r = storage.round_to_bf16(x)
    assert np.all(storage.bf16_bits(r).astype(np.uint32) << 16
                  == r.astype(np.float32).view(np.uint32))       # r is a bf16 number
    pos = r > 0
    dn, up = _bf16_neighbours(np.abs(r))
    err = np.abs(np.abs(x) - np.abs(r))
    assert np.all(err <= np.abs(np.abs(x) - up))
    assert np.all(err <= np.abs(np.abs(x) - dn))
    assert pos.sum() > 1000
    # exact ties go to the even significand
    ties = np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -(2.0 + 2**-7), 2**-126 + 2**-134])
    np.testing.assert_array_equal(storage.round_to_bf16(ties),
                                  [1.0, 1.0 + 2**-6, -2.0, 2**-126])


def test_bf16_overflow_and_specials():
    big = np.array([3.3895313892515355e38, 3.39e38, 3.4e38, 1e300, -1e300, np.inf, -np.inf])
    r = storage.round_to_bf16(big)
    assert r[0] == storage.BF16_MAX
    assert np.isinf(r[2:]).all()
    assert np.isnan(storage.round_to_bf16(np.array([np.nan]))).all()


def test_f32_and_f64_rounding():
    x = np.array([1.0 + 2**-30, 0.1, -7.25])
    np.testing.assert_array_equal(storage.round_to(x, "f64"), x)
    np.testing.assert_array_equal(storage.round_to(x, "f32"), x.astype(np.float32).astype(np.float64))
    with pytest.raises(ValueError):
        storage.round_to(x, "f16")
