"""Host-buffer suffix prefill (kvc_prefill_suffix_host) against the device-buffer call.

The host-buffer entry point copies each stage's rows into device staging, runs
the same append and attention kernels per stage and copies the output rows
back.  Every (sequence, head, query tile) is computed by the same kernel code
from the same inputs, so its results must equal kvc_prefill_suffix's bit for
bit: outputs, stored rows, positions and lengths.  One case is also checked
against the float64 oracle's full masked recomputation ([LCP5] section
"先看一次历史编辑").  A rejected call must leave the cache unchanged ([Ch37]
"Reset or reject without corrupting retained state").
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, device_tensor, need_gpu, storage_np, to_np
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
from oracle import attention as A

pytestmark = pytest.mark.gpu
BASE = 10000.0


def setup_pair(B, Hq, Hkv, D, T, cuts, dtype, block_rows, seed):
    """Two caches holding the same prefix rows, truncated to `cuts`, and the suffix inputs."""
    qd = device_tensor(W.normal_np((B, Hq, T, D), seed), dtype)
    kd = device_tensor(W.normal_np((B, Hkv, T, D), seed + 1), dtype)
    vd = device_tensor(W.normal_np((B, Hkv, T, D), seed + 2), dtype)
    caches = []
    for _ in range(2):
        c = KVCache(B, Hq, T + 16, D, heads_kv=Hkv, dtype=dtype, rope_base=BASE, block_rows=block_rows)
        c.prefill_suffix(0, None, kd, vd, out=False)
        c.truncate(cuts)
        caches.append(c)
    S = max(T - c for c in cuts)
    sel = lambda x: torch.stack([torch.nn.functional.pad(x[b, :, cuts[b]:], (0, 0, 0, S - (T - cuts[b])))
                                 for b in range(B)]).contiguous()
    return caches, (qd, kd, vd), tuple(sel(x) for x in (qd, kd, vd)), [T - c for c in cuts]


def assert_same_state(a, b):
    assert a.get_lengths(0) == b.get_lengths(0)
    for x, y in zip(storage_np(a), storage_np(b)):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("Hq,Hkv,cuts,block_rows,chunk", [
    (4, 4, [150, 0, 257, 300, 60], 0, 0),      # tile kernel; a sequence with no new rows
    (8, 2, [150, 0, 257, 300, 60], 0, 1),      # grouped heads, one sequence per stage
    (8, 2, [1100, 37, 640, 999, 1300], 0, 2),  # many key tiles per query tile, ragged stages
    (4, 1, [150, 0, 257, 300, 60], 64, 3),     # paged storage, single key/value head
])
def test_host_prefill_equals_device_prefill(Hq, Hkv, cuts, block_rows, chunk):
    need_gpu()
    T = 1300 if max(cuts) > 400 else 300
    caches, _, (qs, ks, vs), seqlen = setup_pair(len(cuts), Hq, Hkv, 128, T, cuts, "bf16", block_rows, 70)
    ref = caches[0].prefill_suffix(0, qs, ks, vs, seqlen=seqlen)
    hq, hk, hv = (x.cpu().pin_memory() for x in (qs, ks, vs))
    hout = torch.full(qs.shape, 7.0, dtype=torch.float32).pin_memory()
    caches[1].prefill_suffix_host(0, hq, hk, hv, seqlen=seqlen, out=hout, chunk_sequences=chunk)
    got, want = hout.numpy(), to_np(ref)
    for b, n in enumerate(seqlen):
        np.testing.assert_array_equal(got[b, :, :n], want[b, :, :n])
        assert np.all(got[b, :, n:] == 7.0)          # rows past seqlen are left untouched
    assert_same_state(caches[0], caches[1])
    for c in caches:
        c.check()


def test_host_prefill_matches_oracle():
    need_gpu()
    B, Hq, Hkv, D, T, cuts = 3, 4, 2, 128, 700, [650, 0, 333]
    caches, (qd, kd, vd), (qs, ks, vs), seqlen = setup_pair(B, Hq, Hkv, D, T, cuts, "bf16", 0, 90)
    hout = caches[1].prefill_suffix_host(0, qs.cpu().pin_memory(), ks.cpu().pin_memory(), vs.cpu().pin_memory(),
                                         seqlen=seqlen)
    q, k, v = to_np(qd), to_np(kd), to_np(vd)
    for b in range(B):
        ref = A.suffix_reference(q[b, :, cuts[b]:], k[b], v[b], np.arange(T), cuts[b], BASE, "bf16")
        assert np.abs(hout.numpy()[b, :, :T - cuts[b]] - ref).max() <= TOL["bf16"]
    caches[1].check()


def test_host_prefill_append_only_and_pageable_inputs():
    need_gpu()
    cuts = [100, 0, 250]
    caches, _, (qs, ks, vs), seqlen = setup_pair(3, 4, 2, 128, 300, cuts, "bf16", 0, 110)
    caches[0].prefill_suffix(0, None, ks, vs, seqlen=seqlen, out=False)
    caches[1].prefill_suffix_host(0, None, ks.cpu(), vs.cpu(), seqlen=seqlen, out=None)   # pageable, no output
    assert_same_state(caches[0], caches[1])


def test_host_prefill_f32_generic_kernel():
    need_gpu()
    cuts = [40, 0, 90]
    caches, _, (qs, ks, vs), seqlen = setup_pair(3, 4, 2, 32, 120, cuts, "f32", 0, 130)
    ref = caches[0].prefill_suffix(0, qs, ks, vs, seqlen=seqlen)
    hout = caches[1].prefill_suffix_host(0, qs.cpu(), ks.cpu(), vs.cpu(), seqlen=seqlen, chunk_sequences=2)
    for b, n in enumerate(seqlen):
        np.testing.assert_array_equal(hout.numpy()[b, :, :n], to_np(ref)[b, :, :n])
    assert_same_state(caches[0], caches[1])


def test_host_prefill_rejects_without_change():
    need_gpu()
    cuts = [100, 0, 250]
    caches, _, (qs, ks, vs), seqlen = setup_pair(3, 4, 2, 128, 300, cuts, "bf16", 0, 150)
    c = caches[1]
    before = c.get_lengths(0)
    K0 = storage_np(c)
    hq, hk, hv = (x.cpu().pin_memory() for x in (qs, ks, vs))
    with pytest.raises(KVCError) as e:                 # sequence 0 would exceed the capacity (100 + 300 > 316)
        c.prefill_suffix_host(0, hq, hk, hv, seqlen=[300, seqlen[1], seqlen[2]])
    assert e.value.name == "KVC_ERR_FULL"
    with pytest.raises(KVCError) as e:                 # a negative stage size
        c.prefill_suffix_host(0, hq, hk, hv, seqlen=seqlen, chunk_sequences=-1)
    assert e.value.name == "KVC_ERR_CONFIG"
    # device memory where host memory is expected (the raw C call; the binding refuses it earlier)
    from kv_cache_append_rope_gb300 import _lib as L
    from kv_cache_append_rope_gb300.kvc import host_tensor_desc, tensor_desc
    import ctypes
    st = L.lib.kvc_prefill_suffix_host(c._h, 0, ctypes.byref(host_tensor_desc(hq)), ctypes.byref(tensor_desc(ks)),
                                       ctypes.byref(host_tensor_desc(hv)), None, L.int_array(seqlen), None, 0,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert L.STATUS[st] == "KVC_ERR_CONFIG"
    with pytest.raises(ValueError):                    # the binding refuses CUDA tensors
        c.prefill_suffix_host(0, qs, ks, vs, seqlen=seqlen)
    assert c.get_lengths(0) == before
    for x, y in zip(K0, storage_np(c)):
        np.testing.assert_array_equal(x, y)
    c.check()
