"""kvc_decode_attend_noalloc: the decode entry point for callers that cannot let
a library allocate device memory (an engine that owns all memory through its
own arena, a framework that hands out only its own buffers).  Its output must
match kvc_append_attend's on the same cache, on two calls in a row.

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
