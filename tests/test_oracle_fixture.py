"""Pins of the oracle against the values [Ch37] prints for its fixture."""
import numpy as np

from golden_data import ch37_trace
from oracle import attention as A
from oracle import fixture as F
from oracle.rope import rotate
from kv_cache_append_rope_gb300 import workloads as W


def _replay():
    rows = W.fixture_head_rows()
    cache = A.LayerCache(1, F.H, F.H, F.C, F.DH, "f64", F.ROPE_BASE)
    outs, weights, shapes = [], [], []
    for p in range(3):
        x = rows[p][None]                         # [B=1, H, d_h]; q = k = v
        o = cache.append_attend(x, x, x)
        outs.append(F.merge_heads(o) @ F.head_swap_projection())
        qr = rotate(rows[p], np.full(F.H, p), F.ROPE_BASE)
        weights.append([A.attend_newest(qr[h], cache.logical_keys(0)[h], cache.logical_values(0)[h])[0]
                        for h in range(F.H)])
        shapes.append([1, F.H, int(cache.length[0]), F.DH])
    return cache, outs, weights, shapes


def test_fixture_trace_matches_printed_values():
    rows, outs, shapes, _, _ = ch37_trace()
    cache, my_outs, my_w, my_shapes = _replay()
    assert len(rows) == 12
    for p, h, j, K, V, a in rows:
        np.testing.assert_allclose(cache.K[0, h, j], K, atol=5.1e-10)
        np.testing.assert_allclose(cache.V[0, h, j], V, atol=5.1e-10)
        assert abs(my_w[p][h][j] - a) <= 5.1e-13
    for p in range(3):
        np.testing.assert_allclose(my_outs[p][0], outs[p], atol=5.1e-10)
        assert my_shapes[p] == shapes[p]


def test_fixture_incremental_equals_full_prefix():
    rows = W.fixture_head_rows()
    _, outs, _, _ = _replay()
    for p in range(3):
        hist = np.transpose(rows[:p + 1], (1, 0, 2))          # [H, t, d_h]
        full = A.decode_reference(rows[p], p, hist, hist, np.arange(p + 1), F.ROPE_BASE, "f64")
        y = F.merge_heads(full[None]) @ F.head_swap_projection()
        assert np.abs(y - outs[p]).max() <= 1e-12


def test_fixture_work_counts_and_reset():
    _, _, _, work, reset = ch37_trace()
    full = sum(t for t in range(1, 4))                 # every prefix row projected again
    incremental = 3                                    # one new row per call
    reused = sum(t - 1 for t in range(1, 4))
    assert full == work["full_rows_per_projection"]
    assert incremental == work["incremental_rows_per_projection"]
    assert reused == work["reused_rows_per_kv_projection"]
    assert 2 * reused == work["avoided_rows_across_kv"]
    cache, outs, _, _ = _replay()
    before = int(cache.length[0])
    K, V, Kid = cache.K.copy(), cache.V.copy(), id(cache.K)
    cache.reset()
    assert (before, int(cache.length[0])) == (int(reset["before"]), int(reset["after"]))
    assert id(cache.K) == Kid and np.array_equal(cache.K, K) and np.array_equal(cache.V, V)
    rows = W.fixture_head_rows()
    replay = [F.merge_heads(cache.append_attend(rows[p][None], rows[p][None], rows[p][None]))
              @ F.head_swap_projection() for p in range(3)]
    for a, b in zip(replay, outs):
        np.testing.assert_array_equal(a, b)


def test_random_variant_incremental_equals_full_prefix():
    Wq, Wk, Wv, Wo, x = W.fixture_random_variant(0)
    cache = A.LayerCache(1, F.H, F.H, F.C, F.DH, "f64", F.ROPE_BASE)
    q = F.split_heads(x @ Wq)            # [steps, H, d_h]
    k = F.split_heads(x @ Wk)
    v = F.split_heads(x @ Wv)
    for p in range(3):
        y = F.merge_heads(cache.append_attend(q[p][None], k[p][None], v[p][None])) @ Wo
        assert [1, F.H, int(cache.length[0]), F.DH] == [1, 2, p + 1, 2]
        out = A.decode_reference(q[p], p, np.transpose(k[:p + 1], (1, 0, 2)),
                                 np.transpose(v[:p + 1], (1, 0, 2)), np.arange(p + 1), F.ROPE_BASE, "f64")
        assert np.abs(F.merge_heads(out[None]) @ Wo - y).max() <= 1e-12
