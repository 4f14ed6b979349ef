"""Pins of the sliding-window parts of the oracle.

[LCP5] section "为什么滑窗部分命中必须回退": a window-4 cache over eight tokens
keeps only positions 4..7, so a partial prefix hit cannot reuse it (cut 0) while
a plain append reuses the whole window (cut 8) -- the two window rows of the
table under "27 例得到的计算量与误差" (72 and 24 projected rows).  The windowed
attention (each row sees its W most recent slots) is pinned by its special
cases (W >= t is full attention, W = 1 returns the row's own value) and by a
loop-by-loop evaluation on small inputs.
"""
import math

import numpy as np
import pytest

from golden_data import lcp5_table
from oracle import attention as A
from oracle import prefix as P

CACHED = list(range(1, 9))
TAIL = [9, 10, 11, 12]


def test_window_rows_of_the_table():
    table, _ = lcp5_table()
    queries = {"window_edit_fifth": CACHED[:4] + [20] + CACHED[5:] + TAIL, "window_append": CACHED + TAIL}
    rows = [name for name, row in table.items() if row["policy"] == "window"]
    assert sorted(rows) == sorted(queries)
    for name in rows:
        row, query = table[name], queries[name]
        assert len(query) == row["query_len"]
        cut = P.lcp_cut_window(CACHED, query, 4)
        assert cut == row["cut"], name
        assert P.projection_rows(2, len(query), cut) == row["rows"]
        assert P.projection_rows(2, len(query), 0) == row["full_rows"]


def test_window_rule_edge_cases():
    assert P.lcp_cut_window(CACHED, CACHED, 4) == 0              # no new suffix: recompute
    assert P.lcp_cut_window([], [1, 2], 4) == 0
    assert P.lcp_cut_window(CACHED, CACHED[:7], 4) == 0          # shortened: a partial hit
    assert P.lcp_cut_window(CACHED, CACHED[:4] + [20] + TAIL, 0) == P.lcp_cut(CACHED, CACHED[:4] + [20] + TAIL)
    with pytest.raises(ValueError):
        P.lcp_cut_window(CACHED, [], 4)


def windowed_by_loops(q, K, V, slot, window):
    """One query row against slots max(0, slot - W + 1) .. slot, written with scalar loops."""
    lo = max(0, slot - window + 1) if window else 0
    d = len(q)
    scores = [sum(q[c] * K[j][c] for c in range(d)) / math.sqrt(d) for j in range(lo, slot + 1)]
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    tot = sum(w)
    return [sum(w[jj] * V[lo + jj][c] for jj in range(len(w))) / tot for c in range(d)]


@pytest.mark.parametrize("window", [1, 2, 3, 5, 9])
def test_windowed_attention_by_loops(window):
    rng = np.random.default_rng(window)
    T, d = 9, 4
    Q, K, V = rng.normal(size=(T, d)), rng.normal(size=(T, d)), rng.normal(size=(T, d))
    slots = np.arange(T)
    got = A.causal_attention(Q, K, V, slots, window)
    for i in range(T):
        ref = windowed_by_loops(Q[i].tolist(), K.tolist(), V.tolist(), i, window)
        assert np.abs(got[i] - ref).max() < 1e-12


def test_window_special_cases():
    rng = np.random.default_rng(1)
    T, d = 12, 8
    Q, K, V = rng.normal(size=(T, d)), rng.normal(size=(T, d)), rng.normal(size=(T, d))
    slots = np.arange(T)
    np.testing.assert_array_equal(A.causal_attention(Q, K, V, slots, T), A.causal_attention(Q, K, V, slots))
    np.testing.assert_array_equal(A.causal_attention(Q, K, V, slots, 1), V)
    # decode steps and a suffix chunk agree under the same window
    q = rng.normal(size=(2, 5, d))
    k, v = rng.normal(size=(1, 9, d)), rng.normal(size=(1, 9, d))
    steps = A.decode_steps_reference(np.transpose(q, (1, 0, 2)), k, v, 4, 10000.0, "f64", window=3)
    chunk = A.suffix_reference(q, k, v, np.arange(9), 4, 10000.0, "f64", window=3)
    assert np.abs(np.transpose(steps, (1, 0, 2)) - chunk).max() < 1e-12
