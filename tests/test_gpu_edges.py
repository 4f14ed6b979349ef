"""Edge cases through the C ABI: empty chunks, the capacity and RoPE-position
limits, truncation to zero, the widest head, a batch beyond the fused-step limit."""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, device_tensor, need_gpu, raw_storage_np, storage_np, to_np
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
from oracle import attention as A

pytestmark = pytest.mark.gpu
BASE = 10000.0


def _rows(B, H, T, D, seed, dtype="bf16"):
    return device_tensor(W.normal_np((B, H, T, D), seed), dtype)


def test_empty_chunk_changes_nothing():
    need_gpu()
    B, H, D, C = 2, 4, 128, 64
    cache = KVCache(B, H, C, D)
    k, v, q = _rows(B, H, 8, D, 1), _rows(B, H, 8, D, 2), _rows(B, H, 8, D, 3)
    cache.prefill_suffix(0, q, k, v, seqlen=[5, 3])
    before = raw_storage_np(cache)
    out = cache.prefill_suffix(0, q, k, v, seqlen=[0, 0])
    assert cache.get_lengths(0) == ([5, 3], [5, 3])
    for a, b in zip(before, raw_storage_np(cache)):
        np.testing.assert_array_equal(a, b)
    assert torch.count_nonzero(out).item() == 0
    cache.check()


def test_capacity_boundary_and_position_limit():
    need_gpu()
    B, H, D, C = 1, 2, 128, 130
    cache = KVCache(B, H, C, D)
    k, v, q = _rows(B, H, C + 1, D, 4), _rows(B, H, C + 1, D, 5), _rows(B, H, C + 1, D, 6)
    cache.prefill_suffix(0, None, k[:, :, :C - 1].contiguous(), v[:, :, :C - 1].contiguous(), out=False)
    one = lambda x, i: x[:, :, i:i + 1].contiguous()
    out = to_np(cache.append_attend(0, one(q, C - 1), one(k, C - 1), one(v, C - 1)))  # fills the last slot
    assert cache.get_lengths(0) == ([C], [C])
    ref = A.decode_reference(to_np(q)[0, :, C - 1], C - 1, to_np(k)[0, :, :C], to_np(v)[0, :, :C], np.arange(C),
                             BASE, "bf16")
    assert np.abs(out[0, :, 0] - ref).max() <= TOL["bf16"]
    before = raw_storage_np(cache)
    for call in (lambda: cache.append_attend(0, one(q, C), one(k, C), one(v, C)),
                 lambda: cache.prefill_suffix(0, None, one(k, C), one(v, C), out=False)):
        with pytest.raises(KVCError) as e:
            call()
        assert e.value.name == "KVC_ERR_FULL"
    for a, b in zip(before, raw_storage_np(cache)):
        np.testing.assert_array_equal(a, b)
    # RoPE table of 64 positions: position 63 is the last one, 64 is rejected
    small = KVCache(1, 2, 64, D, rope_max_positions=64)
    small.prefill_suffix(0, None, k[:, :, :4].contiguous(), v[:, :, :4].contiguous(), start_pos=[60], out=False)
    assert small.get_lengths(0) == ([4], [64])
    Ks, _, P = storage_np(small)
    assert P[0, :4].tolist() == [60, 61, 62, 63]
    Kref, _ = A.stored_rows(to_np(k)[0, :, :4], to_np(v)[0, :, :4], (60 + np.arange(4))[None], BASE, "bf16")
    np.testing.assert_array_equal(Ks[0, :, :4], Kref)
    with pytest.raises(KVCError) as e:
        small.append_attend(0, one(q, 4), one(k, 4), one(v, 4))
    assert e.value.name == "KVC_ERR_POSITION"
    assert small.get_lengths(0) == ([4], [64])
    cache.check()
    small.check()


def test_truncate_to_zero_then_decode_from_empty():
    need_gpu()
    B, H, D = 2, 4, 128
    cache = KVCache(B, H, 32, D)
    k, v, q = _rows(B, H, 10, D, 7), _rows(B, H, 10, D, 8), _rows(B, H, 10, D, 9)
    cache.prefill_suffix(0, None, k, v, out=False)
    cache.truncate([0, 0])
    out = to_np(cache.append_attend(0, q[:, :, :1].contiguous(), k[:, :, :1].contiguous(), v[:, :, :1].contiguous()))
    np.testing.assert_allclose(out[:, :, 0], to_np(v)[:, :, 0], atol=1e-6)     # t = 1: the value itself
    assert cache.get_lengths(0) == ([1, 1], [1, 1])
    cache.check()


@pytest.mark.parametrize("D", [256, 8])
def test_head_width_extremes_generic_path(D):
    need_gpu()
    B, H, L0 = 2, 2, [3, 40]
    T = max(L0) + 1
    k, v, q = _rows(B, H, T, D, 10), _rows(B, H, T, D, 11), _rows(B, H, T, D, 12)
    cache = KVCache(B, H, 64, D)
    cache.prefill_suffix(0, None, k[:, :, :max(L0)].contiguous(), v[:, :, :max(L0)].contiguous(), seqlen=L0,
                         out=False)
    idx = torch.tensor(L0, device="cuda")
    sel = lambda x: x[torch.arange(B, device="cuda"), :, idx][:, :, None, :].contiguous()
    out = to_np(cache.append_attend(0, sel(q), sel(k), sel(v)))
    kn, vn, qn = to_np(k), to_np(v), to_np(q)
    for b in range(B):
        n = L0[b] + 1
        ref = A.decode_steps_reference(qn[b, :, L0[b]][None], kn[b, :, :n], vn[b, :, :n], L0[b], BASE, "bf16")
        assert np.abs(out[b, :, 0] - ref[0]).max() <= TOL["bf16"]


def test_batch_beyond_fused_step_limit():
    """B = 300 > 256 sequences: the separate-kernel step serves it."""
    need_gpu()
    B, H, D = 300, 1, 128
    rng = np.random.default_rng(13)
    L0 = rng.integers(1, 100, B).tolist()
    T = max(L0) + 1
    k, v, q = _rows(B, H, T, D, 14), _rows(B, H, T, D, 15), _rows(B, H, T, D, 16)
    cache = KVCache(B, H, 128, D)
    cache.prefill_suffix(0, None, k[:, :, :max(L0)].contiguous(), v[:, :, :max(L0)].contiguous(), seqlen=L0,
                         out=False)
    idx = torch.tensor(L0, device="cuda")
    sel = lambda x: x[torch.arange(B, device="cuda"), :, idx][:, :, None, :].contiguous()
    out = to_np(cache.append_attend(0, sel(q), sel(k), sel(v)))
    kn, vn, qn = to_np(k), to_np(v), to_np(q)
    for b in [0, 1, 150, 299]:
        n = L0[b] + 1
        ref = A.decode_steps_reference(qn[b, :, L0[b]][None], kn[b, :, :n], vn[b, :, :n], L0[b], BASE, "bf16")
        assert np.abs(out[b, :, 0] - ref[0]).max() <= TOL["bf16"]
    assert cache.get_lengths(0)[0] == [l + 1 for l in L0]
    cache.check()
