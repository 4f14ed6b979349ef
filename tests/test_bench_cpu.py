"""Host-side pieces of bench.py that need no GPU: the one-thread oracle timing used for
`cpu_baseline.one_core` runs the oracle in a fresh interpreter limited to one BLAS/OpenMP
thread and returns its time; the result it times is the oracle's own (same call)."""
import sys

import numpy as np


def _bench():
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        import bench
    finally:
        sys.argv = argv
    return bench


def test_one_thread_oracle_timing_runs_both_calls():
    bench = _bench()
    rng = np.random.default_rng(0)
    L0, steps, G = 200, 4, 4
    k = rng.standard_normal((1, L0 + steps, 128))
    v = rng.standard_normal((1, L0 + steps, 128))
    q = rng.standard_normal((steps, G, 128))
    s = bench.oracle_seconds_one_thread("decode", {"q": q, "k": k, "v": v, "L0": np.int64(L0)})
    assert 0.0 < s < 60.0
    T, cut = 400, 300
    arrays = {"q": rng.standard_normal((1, T - cut, 128)), "k": rng.standard_normal((1, T, 128)),
              "v": rng.standard_normal((1, T, 128)), "T": np.int64(T), "cut": np.int64(cut),
              "rows": np.arange(0, T - cut, 9)}
    s = bench.oracle_seconds_one_thread("suffix", arrays)
    assert 0.0 < s < 60.0
