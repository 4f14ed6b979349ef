"""The chapter-37 fixture through libkvc (f64): printed values, reset, and the
rejected calls of its error evidence, each leaving the cache unchanged."""
import ctypes

import numpy as np
import pytest
import torch

from golden_data import ch37_trace
from gpu_helpers import need_gpu, raw_storage_np, storage_np, to_np
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
from oracle import attention as A
from oracle import fixture as F

pytestmark = pytest.mark.gpu


def _rows_dev(p):
    rows = W.fixture_head_rows()
    return torch.from_numpy(rows[p]).reshape(1, 2, 1, 2).to("cuda", torch.float64).contiguous()


def _swap(o):
    return to_np(o).reshape(1, 4) @ F.head_swap_projection()


def test_fixture_trace_and_reset():
    need_gpu()
    rows, outs, shapes, _, reset = ch37_trace()
    cache = KVCache(1, 2, 4, 2, dtype="f64", rope_base=10000.0)
    got = []
    for p in range(3):
        x = _rows_dev(p)
        got.append(_swap(cache.append_attend(0, x, x, x)))
        assert cache.get_lengths(0)[0] == [p + 1]
    for p in range(3):
        np.testing.assert_allclose(got[p][0], outs[p], atol=5.1e-10)
    K, V, P = storage_np(cache)
    for p, h, j, Kp, Vp, _ in rows:
        np.testing.assert_allclose(K[0, h, j], Kp, atol=5.1e-10)
        np.testing.assert_allclose(V[0, h, j], Vp, atol=5.1e-10)
    assert P[0, :3].tolist() == [0, 1, 2]
    # incremental == full prefix (oracle) within 1e-12
    hr = W.fixture_head_rows()
    for p in range(3):
        hist = np.transpose(hr[:p + 1], (1, 0, 2))
        ref = A.decode_reference(hr[p], p, hist, hist, np.arange(p + 1), 10000.0, "f64")
        assert np.abs(ref.reshape(1, 4) @ F.head_swap_projection() - got[p]).max() <= 1e-12
    # reset: length 0, same allocation, bytes unchanged, identical replay
    ptr_before = cache.storage(0)[0].data_ptr()
    before = raw_storage_np(cache)
    cache.reset()
    assert cache.get_lengths(0) == ([0], [0]) and cache.get_len(0) == [0]
    after = raw_storage_np(cache)
    assert cache.storage(0)[0].data_ptr() == ptr_before
    for a, b in zip(before, after):
        np.testing.assert_array_equal(a, b)
    # the logical snapshot holds no row after a reset
    K0, V0, P0 = storage_np(cache)
    assert not K0.any() and not V0.any() and (P0 == -1).all()
    replay = [_swap(cache.append_attend(0, _rows_dev(p), _rows_dev(p), _rows_dev(p))) for p in range(3)]
    for a, b in zip(replay, got):
        np.testing.assert_array_equal(a, b)
    assert int(reset["before"]) == 3 and int(reset["after"]) == 0
    cache.check()


def test_random_variant_incremental_equals_full_prefix():
    need_gpu()
    Wq, Wk, Wv, Wo, x = W.fixture_random_variant(0)
    t = lambda a: torch.from_numpy(a).to("cuda", torch.float64)
    cache = KVCache(1, 2, 4, 2, dtype="f64", rope_base=10000.0)
    xd = t(x)
    q = (xd @ t(Wq)).reshape(3, 1, 2, 1, 2)
    k = (xd @ t(Wk)).reshape(3, 1, 2, 1, 2)
    v = (xd @ t(Wv)).reshape(3, 1, 2, 1, 2)
    qn, kn, vn = (to_np(a).reshape(3, 2, 2) for a in (q, k, v))
    for p in range(3):
        y = to_np(cache.append_attend(0, q[p].contiguous(), k[p].contiguous(), v[p].contiguous())).reshape(1, 4) @ Wo
        ref = A.decode_reference(qn[p], p, np.transpose(kn[:p + 1], (1, 0, 2)), np.transpose(vn[:p + 1], (1, 0, 2)),
                                 np.arange(p + 1), 10000.0, "f64").reshape(1, 4) @ Wo
        assert np.abs(y - ref).max() <= 1e-12
        K, V, _ = cache.storage(0)
        assert list(K[:, :, :p + 1].shape) == [1, 2, p + 1, 2]


def _state(cache):
    K, V, P = raw_storage_np(cache)
    return K.copy(), V.copy(), P.copy(), cache.get_lengths(0)


def _unchanged(cache, before):
    after = _state(cache)
    for a, b in zip(before[:3], after[:3]):
        np.testing.assert_array_equal(a, b)
    assert before[3] == after[3]


def test_rejected_calls_leave_the_cache_unchanged():
    need_gpu()
    x = _rows_dev(0)
    cache = KVCache(1, 2, 4, 2, dtype="f64", rope_base=10000.0, checked=True)
    cache.append_attend(0, x, x, x)
    before = _state(cache)
    cases = {
        "two_tokens": (torch.zeros(1, 2, 2, 2, dtype=torch.float64, device="cuda"), x, x, "KVC_ERR_QUERY_SHAPE"),
        "model_width": (torch.zeros(1, 2, 1, 4, dtype=torch.float64, device="cuda"), x, x, "KVC_ERR_QUERY_SHAPE"),
        "head_count_key": (x, torch.zeros(1, 1, 1, 2, dtype=torch.float64, device="cuda"), x, "KVC_ERR_KEY_SHAPE"),
        "head_count_value": (x, x, torch.zeros(1, 1, 1, 2, dtype=torch.float64, device="cuda"), "KVC_ERR_VALUE_SHAPE"),
        "dtype": (x.float(), x, x, "KVC_ERR_DTYPE"),
        "nonfinite_key": (x, torch.full_like(x, float("inf")), x, "KVC_ERR_NONFINITE_KEY"),
        "nonfinite_value": (x, x, torch.full_like(x, float("nan")), "KVC_ERR_NONFINITE_VALUE"),
    }
    for name, (q, k, v, code) in cases.items():
        with pytest.raises(KVCError) as e:
            cache.append_attend(0, q, k, v)
        assert e.value.name == code, name
        _unchanged(cache, before)
    with pytest.raises(KVCError) as e:
        cache.append_attend(1, x, x, x)
    assert e.value.name == "KVC_ERR_LAYER"
    _unchanged(cache, before)
    # full cache: capacity 1, one append, then a second
    small = KVCache(1, 2, 1, 2, dtype="f64", rope_base=10000.0)
    small.append_attend(0, x, x, x)
    before = _state(small)
    with pytest.raises(KVCError) as e:
        small.append_attend(0, x, x, x)
    assert e.value.name == "KVC_ERR_FULL"
    _unchanged(small, before)
    # capacity beyond the RoPE position table
    with pytest.raises(KVCError) as e:
        KVCache(1, 2, 5, 2, dtype="f64", rope_base=10000.0, rope_max_positions=4)
    assert e.value.name == "KVC_ERR_CAPACITY_EXCEEDS_POSITIONS"
    # host memory is refused before any kernel sees it
    with pytest.raises(ValueError):
        cache.append_attend(0, x.cpu(), x, x)
    cache.check()
    small.check()
