"""Can the GPU parity checks fail?  A CPU calibration of the relative-error guard.

At long contexts the attention output is small (|o| ~ t^-1/2 for random rows), so
the contract tolerance of 2e-2 max-abs cannot see a dropped 64-row key tile at
t = 8000 (a change of ~0.009).  The GPU tests therefore also bound the relative
error of every output row, ||got - ref|| / ||ref||, by ``REL_GUARD`` (a
regression guard at the observed error scale, not the contract).  This file
shows, on the CPU, that the guard separates honest results from broken ones:

* honest: the oracle's output with the roundings the bf16 kernels make --
  the rotated, scaled query rounded to bf16, the exponentials rounded to bf16
  before they weight the values (the sum taken from the unrounded ones) -- stays
  well below the guard at every context length the workloads use;
* broken: the same computation with one 64-row key tile dropped, with one
  split's partial result merged twice, or with one poisoned row past the length
  attended (keys 0, values 1e4, as KVC_OPT_TEST_POISON writes them), lands far
  above it -- and a dropped tile at t >= 4000 passes the 2e-2 max-abs contract,
  which is why the guard exists.
The emulation is test code (it shares nothing with the CUDA path); the exact
result is the oracle's.
"""
import math

import numpy as np
import pytest

from gpu_helpers_cpu import REL_GUARD, rel_err
from oracle import attention as A
from oracle.storage import round_to_bf16

D = 128
LOG2E = 1.4426950408889634


def _lane(t, seed):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=D)
    K = round_to_bf16(rng.normal(size=(t, D)))
    V = round_to_bf16(rng.normal(size=(t, D)))
    return q, K, V


def _bf16_kernel_like(q, K, V, keep=None, twice=None):
    """Attention with the bf16 kernels' roundings; `keep` masks keys out, `twice`
    counts a range of keys (one split) twice."""
    qb = round_to_bf16(q * (LOG2E / math.sqrt(D)))
    s = K @ qb                                   # log2 units
    w = np.ones(len(s))
    if keep is not None:
        w = w * keep
    if twice is not None:
        w[twice] += 1.0
    m = s[w > 0].max()
    p = np.exp2(s - m) * w
    pb = round_to_bf16(np.exp2(s - m)) * w
    return (pb @ V) / p.sum()


@pytest.mark.parametrize("t", [300, 1000, 4000, 8000, 16896, 32767])
def test_guard_separates_honest_from_broken_results(t):
    q, K, V = _lane(t, seed=t)
    exact = A.attend_newest(q, K, V)[1]
    honest = _bf16_kernel_like(q, K, V)
    assert rel_err(honest, exact) < REL_GUARD / 3
    # one 64-row tile in the middle of the keys dropped
    keep = np.ones(t)
    a = (t // 2) // 64 * 64
    keep[a:a + 64] = 0
    dropped = _bf16_kernel_like(q, K, V, keep=keep)
    assert rel_err(dropped, exact) > 2 * REL_GUARD
    if t >= 4000:
        assert np.abs(dropped - exact).max() < 2e-2      # the contract alone would pass it
    # a split of 256 rows (the smallest automatic split) merged twice
    twice = np.zeros(t, dtype=bool)
    twice[a:a + 256] = True
    doubled = _bf16_kernel_like(q, K, V, twice=twice)
    assert rel_err(doubled, exact) > 2 * REL_GUARD


@pytest.mark.parametrize("t", [300, 8000, 32767])
def test_one_poisoned_row_is_far_beyond_the_guard(t):
    q, K, V = _lane(t, seed=t + 1)
    exact = A.attend_newest(q, K, V)[1]
    Kp = np.vstack([K, np.zeros((1, D))])
    Vp = np.vstack([V, np.full((1, D), 9984.0)])     # 1e4 in bf16
    leaked = A.attend_newest(q, Kp, Vp)[1]
    assert rel_err(leaked, exact) > 10 * REL_GUARD
    assert np.abs(leaked - exact).max() > 2e-2        # the contract sees it too


def test_guard_statistic():
    assert rel_err(np.array([1.0, 0.0]), np.array([1.0, 0.0])) == 0.0
    assert abs(rel_err(np.array([[1.1, 0.0], [0.0, 2.0]]), np.array([[1.0, 0.0], [0.0, 2.0]])) - 0.1) < 1e-12
