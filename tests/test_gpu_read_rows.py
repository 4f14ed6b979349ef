"""kvc_read_rows and kvc_get_len: the logical snapshot of a layer ([Ch37] listing
"Own a fixed layer-bound cache, append one checked row, and reset logical
length": keys() / values() return the retained rows, never the unused capacity).

Stored rows are compared bit for bit with the oracle's definition of what an
append writes (``oracle.attention.stored_rows``: the key rotated at its
position in float64 and rounded once to the storage dtype, the value rounded),
for contiguous and paged storage (blocks shared between sequences included),
every storage dtype and both copy widths of the gather kernel (rows that are a
multiple of 16 bytes and rows that are not).  Rows at or past a length must
read as zero with position -1.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import device_tensor, need_gpu, to_np
from kv_cache_append_rope_gb300 import _lib as L
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
from oracle import attention as A

pytestmark = pytest.mark.gpu
BASE = 10000.0


def _check_snapshot(cache, k, v, lens, R=None, layer=0):
    """k, v: unrotated rows [B, H_kv, T, d] (float64, storage-dtype values); row j at position j."""
    dtype = {0: "bf16", 1: "f32", 2: "f64"}[cache.config.dtype]
    Ks, Vs, Ps = cache.read_rows(layer, rows=R)
    Ks, Vs, Ps = to_np(Ks), to_np(Vs), Ps.cpu().numpy()
    R = Ks.shape[2]
    for b, n in enumerate(lens):
        m = min(n, R)
        K, V = A.stored_rows(k[b, :, :m], v[b, :, :m], np.arange(m)[None], BASE, dtype)
        np.testing.assert_array_equal(Ks[b, :, :m], K)
        np.testing.assert_array_equal(Vs[b, :, :m], V)
        assert Ps[b, :m].tolist() == list(range(m))
        assert not Ks[b, :, m:].any() and not Vs[b, :, m:].any()
        assert (Ps[b, m:] == -1).all()
    assert cache.get_len(layer) == list(lens) == cache.get_lengths(layer)[0]


@pytest.mark.parametrize("dtype,D,block_rows", [("bf16", 128, 0), ("bf16", 128, 64), ("f32", 6, 0),
                                                ("f64", 16, 128), ("bf16", 2, 0)])
def test_snapshot_equals_the_oracle_rows(dtype, D, block_rows):
    need_gpu()
    B, Hq, Hkv, C = 3, 4, 2, 300
    L0 = [0, 130, 257]
    steps = 3
    T = max(L0) + steps
    kd = device_tensor(W.normal_np((B, Hkv, T, D), 11), dtype)
    vd = device_tensor(W.normal_np((B, Hkv, T, D), 12), dtype)
    qd = device_tensor(W.normal_np((B, Hq, T, D), 13), dtype)
    cache = KVCache(B, Hq, C, D, heads_kv=Hkv, dtype=dtype, block_rows=block_rows)
    cache.prefill_suffix(0, None, kd[:, :, :max(L0)].contiguous(), vd[:, :, :max(L0)].contiguous(), seqlen=L0,
                         out=False)
    k, v = to_np(kd), to_np(vd)
    _check_snapshot(cache, k, v, L0)
    for s in range(steps):
        idx = torch.tensor([l + s for l in L0], device="cuda")
        sel = lambda x: x[torch.arange(B, device="cuda"), :, idx][:, :, None, :].contiguous()
        cache.append_attend(0, sel(qd), sel(kd), sel(vd))
    # sequence b now holds rows 0 .. L0[b] + steps - 1, its decode rows at L0[b] .. : rebuild
    # its unrotated history in slot order for the oracle
    hist_k = np.zeros((B, Hkv, T, D))
    hist_v = np.zeros((B, Hkv, T, D))
    for b, l0 in enumerate(L0):
        hist_k[b, :, :l0 + steps] = k[b, :, :l0 + steps]
        hist_v[b, :, :l0 + steps] = v[b, :, :l0 + steps]
    lens = [l + steps for l in L0]
    _check_snapshot(cache, hist_k, hist_v, lens)
    _check_snapshot(cache, hist_k, hist_v, lens, R=200)          # a shorter snapshot: rows < R only
    # truncate: rows past the cut leave the snapshot although their bytes stay in storage
    cache.truncate([2, 64, 100])
    _check_snapshot(cache, hist_k, hist_v, [2, 64, 100])
    cache.check()


def test_snapshot_of_shared_blocks_and_copy_on_write():
    need_gpu()
    B, H, D, C, P = 2, 2, 128, 512, 64
    T = 200
    kd = device_tensor(W.normal_np((B, H, T + 8, D), 21), "bf16")
    vd = device_tensor(W.normal_np((B, H, T + 8, D), 22), "bf16")
    qd = device_tensor(W.normal_np((B, H, T + 8, D), 23), "bf16")
    cache = KVCache(B, H, C, D, block_rows=P)
    # sequence 0 holds T rows, sequence 1 none; then 1 shares 0's first 150 rows
    cache.prefill_suffix(0, None, kd[:, :, :T].contiguous(), vd[:, :, :T].contiguous(), seqlen=[T, 0], out=False)
    cache.share_prefix(1, 0, 150)
    k, v = to_np(kd), to_np(vd)
    hist_k = np.stack([k[0], k[0]])
    hist_v = np.stack([v[0], v[0]])
    _check_snapshot(cache, hist_k, hist_v, [T, 150])
    # a decode step writes into sequence 1's partly filled shared block: it is copied first
    x = lambda t, b: t[:, :, T:T + 1].contiguous()
    cache.append_attend(0, x(qd, 0), x(kd, 0), x(vd, 0))
    hist_k[0, :, T] = k[0, :, T]
    hist_v[0, :, T] = v[0, :, T]
    hist_k[1, :, 150] = k[1, :, T]
    hist_v[1, :, 150] = v[1, :, T]
    # sequence 1's new row sits at slot 150 but was rotated at position 150: rebuild it
    Ks, Vs, Ps = cache.read_rows(0)
    Ks, Vs = to_np(Ks), to_np(Vs)
    K1, V1 = A.stored_rows(k[1, :, T:T + 1], v[1, :, T:T + 1], np.array([[150]]), BASE, "bf16")
    np.testing.assert_array_equal(Ks[1, :, 150:151], K1)
    np.testing.assert_array_equal(Vs[1, :, 150:151], V1)
    K0, V0 = A.stored_rows(hist_k[0, :, :T + 1], hist_v[0, :, :T + 1], np.arange(T + 1)[None], BASE, "bf16")
    np.testing.assert_array_equal(Ks[0, :, :T + 1], K0)
    np.testing.assert_array_equal(Ks[1, :, :150], K0[:, :150])      # the shared rows are still the source's
    assert not Ks[1, :, 151:].any()
    cache.check()


def test_snapshot_follows_device_length_steps_without_a_sync():
    need_gpu()
    B, H, D, C = 2, 4, 128, 256
    L0 = [5, 70]
    T = max(L0) + 2
    kd = device_tensor(W.normal_np((B, H, T, D), 31), "bf16")
    vd = device_tensor(W.normal_np((B, H, T, D), 32), "bf16")
    qd = device_tensor(W.normal_np((B, H, T, D), 33), "bf16")
    cache = KVCache(B, H, C, D)
    cache.prefill_suffix(0, None, kd[:, :, :max(L0)].contiguous(), vd[:, :, :max(L0)].contiguous(), seqlen=L0,
                         out=False)
    cache.set_option(L.OPT_DEVICE_LENGTHS, 1)
    idx = torch.tensor(L0, device="cuda")
    sel = lambda x: x[torch.arange(B, device="cuda"), :, idx][:, :, None, :].contiguous()
    cache.append_attend(0, sel(qd), sel(kd), sel(vd))
    Ks, _, Ps = cache.read_rows(0)          # stream-ordered after the step: sees its rows
    Ps = Ps.cpu().numpy()
    for b, l0 in enumerate(L0):
        assert Ps[b, :l0 + 1].tolist() == list(range(l0 + 1)) and Ps[b, l0 + 1] == -1
        K, _ = A.stored_rows(to_np(kd)[b, :, :l0 + 1], to_np(vd)[b, :, :l0 + 1], np.arange(l0 + 1)[None], BASE,
                             "bf16")
        np.testing.assert_array_equal(to_np(Ks)[b, :, :l0 + 1], K)
    cache.set_option(L.OPT_DEVICE_LENGTHS, 0)
    cache.check()


def test_snapshot_rejects_bad_arguments():
    need_gpu()
    cache = KVCache(2, 2, 64, 16, dtype="f32")
    for rows, code in ((65, "KVC_ERR_KEY_SHAPE"), (0, "KVC_ERR_KEY_SHAPE")):
        with pytest.raises(KVCError) as e:
            cache.read_rows(0, rows=rows)
        assert e.value.name == code
    with pytest.raises(KVCError) as e:
        cache.read_rows(3)
    assert e.value.name == "KVC_ERR_LAYER"
    from kv_cache_append_rope_gb300.kvc import tensor_desc, _stream
    import ctypes
    wrong = torch.zeros((2, 2, 64, 16), dtype=torch.float64, device="cuda")
    d = tensor_desc(wrong)
    st = L.lib.kvc_read_rows(cache._h, 0, ctypes.byref(d), None, None, _stream(None))
    assert L.STATUS[st] == "KVC_ERR_DTYPE"
    cache.check()
