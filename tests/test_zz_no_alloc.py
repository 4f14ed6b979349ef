"""kvc_decode_attend_noalloc: the decode entry point for callers that cannot let
a library allocate device memory (an engine that owns all memory through its
own arena, a framework that hands out only its own buffers).  Its output must
match kvc_append_attend's on the same cache, on two calls in a row, and the
float64 oracle's on caches built from the oracle's own stored rows: MHA/GQA,
32 query heads per key/value head with several splits (the separate merge
launch), and a batch whose partials only fit the static array once the split
plan is widened.  kvc_noalloc_check must report a bounded wait that gave up.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, device_tensor, need_gpu
from kv_cache_append_rope_gb300 import _lib as L
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, _stream
from oracle import attention as A
from oracle import rope as R

pytestmark = pytest.mark.gpu


def rotate_queries(q, positions, base=10000.0):
    """Rotated f32 queries [B, H_q, 128] for the new entry point (torch, float64 on the GPU)."""
    B, H, _, D = q.shape
    x = q[:, :, 0].to(torch.float64)
    j = torch.arange(D // 2, dtype=torch.float64, device=q.device)
    theta = torch.pow(torch.tensor(base, dtype=torch.float64, device=q.device), -(2.0 * j) / D)
    ang = torch.as_tensor(positions, dtype=torch.float64, device=q.device)[:, None, None] * theta
    c, s = torch.cos(ang), torch.sin(ang)
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = torch.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out.to(torch.float32).contiguous()


def call_noalloc(K, V, q_rot, lengths, out, B, Hq, Hkv, C):
    return L.STATUS[L.lib.kvc_decode_attend_noalloc(
        K.data_ptr(), V.data_ptr(), q_rot.data_ptr(), L.int_array(lengths), out.data_ptr(),
        B, Hq, Hkv, C, _stream(None))]


def test_noalloc_decode_matches_append_attend_twice():
    need_gpu()
    B, Hq, Hkv, D, C = 3, 8, 2, 128, 700
    L0 = [1, 200, 517]
    steps = 2
    T = max(L0) + steps
    kd = device_tensor(W.normal_np((B, Hkv, T, D), 91), "bf16")
    vd = device_tensor(W.normal_np((B, Hkv, T, D), 92), "bf16")
    qd = device_tensor(W.normal_np((B, Hq, T, D), 93), "bf16")
    cache = KVCache(B, Hq, C, D, heads_kv=Hkv, dtype="bf16")
    cache.prefill_suffix(0, None, kd[:, :, :max(L0)].contiguous(), vd[:, :, :max(L0)].contiguous(),
                         seqlen=L0, out=False)
    K, V, _ = cache.storage(0)
    for step in range(steps):
        idx = torch.tensor([l + step for l in L0], device="cuda")
        sel = lambda x: x[torch.arange(B, device="cuda"), :, idx][:, :, None, :].contiguous()
        q = sel(qd)
        ref = cache.append_attend(0, q, sel(kd), sel(vd))[:, :, 0]
        lengths = [l + step + 1 for l in L0]
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        st = call_noalloc(K, V, rotate_queries(q, [l + step for l in L0]), lengths, out, B, Hq, Hkv, C)
        assert st == "KVC_OK"
        torch.cuda.synchronize()
        err = (out - ref).abs().max().item()
        assert err <= TOL["bf16"], err


def test_noalloc_rejects_sizes_beyond_its_scratch():
    need_gpu()
    K = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(16, dtype=torch.float32, device="cuda")
    assert call_noalloc(K, K, q, [5], q, 1, 8, 2, 4) == "KVC_ERR_FULL"            # length beyond capacity
    assert call_noalloc(K, K, q, [0], q, 1, 8, 2, 4) == "KVC_ERR_FULL"            # empty sequence
    assert call_noalloc(K, K, q, [1] * 600, q, 600, 32, 8, 4) == "KVC_ERR_CONFIG"  # B * H_q beyond the array
    assert call_noalloc(K, K, q, [1], q, 1, 64, 1, 4) == "KVC_ERR_CONFIG"         # more than 32 heads per group


def _oracle_case(B, Hq, Hkv, C, lengths, seed):
    """Caller-owned cache built from the oracle's stored rows, rotated f32 queries, and
    the oracle's outputs [B, H_q, 128] for the sequences in ``check``."""
    D = 128
    rng = np.random.default_rng(seed)
    k = rng.normal(size=(B, Hkv, C, D))
    v = rng.normal(size=(B, Hkv, C, D))
    K, V = A.stored_rows(k, v, np.arange(C)[None, None], 10000.0, "bf16")
    q = rng.normal(size=(B, Hq, D))
    pos = np.asarray(lengths) - 1
    qr = R.rotate(q, np.broadcast_to(pos[:, None], (B, Hq)), 10000.0)
    qr32 = qr.astype(np.float32)
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dt)
    return dev(K, torch.bfloat16), dev(V, torch.bfloat16), dev(qr32, torch.float32), K, V, qr32


def _oracle_out(K, V, qr, lengths, Hq, Hkv, b):
    out = np.empty((Hq, 128))
    for h in range(Hq):
        g = A.kv_head_of(h, Hq, Hkv)
        out[h] = A.attend_newest(qr[b, h].astype(np.float64), K[b, g, :lengths[b]], V[b, g, :lengths[b]])[1]
    return out


def _check():
    return L.STATUS[L.lib.kvc_noalloc_check(_stream(None))]


@pytest.mark.parametrize("B,Hq,Hkv,C,lengths", [
    (3, 8, 2, 700, [1, 200, 517]),                   # GQA, one split each
    (4, 32, 1, 3072, [3000, 1, 2047, 2900]),         # 32 heads per group, many splits + merge launch
])
def test_noalloc_matches_the_oracle_twice(B, Hq, Hkv, C, lengths):
    need_gpu()
    Kd, Vd, qd, K, V, qr = _oracle_case(B, Hq, Hkv, C, lengths, seed=B * 100 + Hq)
    for _ in range(2):
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        assert call_noalloc(Kd, Vd, qd, lengths, out, B, Hq, Hkv, C) == "KVC_OK"
        got = out.double().cpu().numpy()
        for b in range(B):
            err = np.abs(got[b] - _oracle_out(K, V, qr, lengths, Hq, Hkv, b)).max()
            assert err <= TOL["bf16"], (b, err)
    assert _check() == "KVC_OK"


def test_noalloc_widened_split_plan_matches_the_oracle():
    """B * H_q = 16000 query heads: the partials of the automatic split plan do not fit
    the static array, so the plan is widened until they do (one split per sequence)."""
    need_gpu()
    B, Hq, Hkv, C, D = 500, 32, 1, 2048, 128
    rng = np.random.default_rng(7)
    lengths = rng.integers(1000, C + 1, size=B).tolist()
    # build the cache on the device (the oracle rows of the sampled sequences are rebuilt below)
    k = W.normal((B, Hkv, C, D), 71, dtype=torch.float64)
    v = W.normal((B, Hkv, C, D), 72, dtype=torch.float64)
    q = W.normal((B, Hq, D), 73, dtype=torch.float64)
    check = [0, 1, int(np.argmax(lengths)), int(np.argmin(lengths)), 250, 499]
    Ks, Vs, qrs = {}, {}, {}
    Kd = torch.empty((B, Hkv, C, D), dtype=torch.bfloat16, device="cuda")
    Vd = torch.empty_like(Kd)
    qd = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    for b in range(B):
        kb, vb = k[b].cpu().numpy(), v[b].cpu().numpy()
        Kb, Vb = A.stored_rows(kb, vb, np.arange(C)[None], 10000.0, "bf16")
        qb = R.rotate(q[b].cpu().numpy(), np.full(Hq, lengths[b] - 1), 10000.0).astype(np.float32)
        Kd[b] = torch.from_numpy(Kb).to(torch.bfloat16)
        Vd[b] = torch.from_numpy(Vb).to(torch.bfloat16)
        qd[b] = torch.from_numpy(qb)
        if b in check:
            Ks[b], Vs[b], qrs[b] = Kb, Vb, qb
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    assert call_noalloc(Kd, Vd, qd, lengths, out, B, Hq, Hkv, C) == "KVC_OK"
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    for b in check:
        ref = np.stack([A.attend_newest(qrs[b][h].astype(np.float64), Ks[b][0, :lengths[b]],
                                        Vs[b][0, :lengths[b]])[1] for h in range(Hq)])
        err = np.abs(got[b] - ref).max()
        assert err <= TOL["bf16"], (b, err)
    assert _check() == "KVC_OK"


def test_noalloc_reports_a_wait_that_gave_up():
    """A planted stall (the producer issues no loads; the consumers' bounded waits give up
    after about a second) is reported by kvc_noalloc_check, once; the next call is sound."""
    need_gpu()
    B, Hq, Hkv, C = 2, 8, 2, 256
    lengths = [100, 256]
    Kd, Vd, qd, K, V, qr = _oracle_case(B, Hq, Hkv, C, lengths, seed=5)
    out = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
    assert _check() == "KVC_OK"
    assert L.STATUS[L.lib.kvc_set_option(None, L.OPT_TEST_STALL, 1)] == "KVC_OK"
    assert call_noalloc(Kd, Vd, qd, lengths, out, B, Hq, Hkv, C) == "KVC_OK"   # enqueued; fails on the device
    assert _check() == "KVC_ERR_DEVICE"
    assert _check() == "KVC_OK"                                               # reported once
    assert call_noalloc(Kd, Vd, qd, lengths, out, B, Hq, Hkv, C) == "KVC_OK"
    assert _check() == "KVC_OK"
    got = out.double().cpu().numpy()
    for b in range(B):
        assert np.abs(got[b] - _oracle_out(K, V, qr, lengths, Hq, Hkv, b)).max() <= TOL["bf16"]
