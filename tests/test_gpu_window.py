"""Sliding-window attention through libkvc against the float64 oracle.

[LCP5] section "为什么滑窗部分命中必须回退": a window-W cache serves each row its W
most recent rows (a window of 4 over eight tokens keeps positions 4..7), and a
partial prefix hit of a window cache is recomputed while a full hit with new
tokens reuses it.  The kvc_config window applies that attention to decode steps
(fused, separate, device-length and generic kernels) and suffix chunks (tile and
generic kernels); kvc_lcp_window applies the reuse rule.  Stored rows, positions
and lengths bit-exact; outputs within 1e-12 (f64), 1e-5 (f32), 2e-2 (bf16).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, TOL, device_tensor, need_gpu, storage_np, to_np
from kv_cache_append_rope_gb300 import _lib as L
from kv_cache_append_rope_gb300 import kvc
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache
from oracle import attention as A
from oracle import prefix as P
from oracle.toy_decoder import ToyDecoder

pytestmark = pytest.mark.gpu
BASE = 10000.0


def inputs(B, Hq, Hkv, T, D, dtype, seed):
    return (device_tensor(W.normal_np((B, Hq, T, D), seed), dtype),
            device_tensor(W.normal_np((B, Hkv, T, D), seed + 1), dtype),
            device_tensor(W.normal_np((B, Hkv, T, D), seed + 2), dtype))


@pytest.mark.parametrize("dtype,D,Hq,Hkv,mode,window", [
    ("bf16", 128, 8, 2, "fused", 100),
    ("bf16", 128, 8, 2, "fused", 64),
    ("bf16", 128, 8, 2, "fused", 1),
    ("bf16", 128, 32, 1, "fused", 300),
    ("bf16", 128, 8, 2, "separate", 100),
    ("bf16", 128, 8, 2, "device", 100),
    ("bf16", 128, 4, 4, "splits", 200),
    ("f64", 16, 4, 2, "generic", 50),
    ("f32", 64, 4, 4, "generic", 7),
])
def test_windowed_decode_matches_oracle(dtype, D, Hq, Hkv, mode, window):
    need_gpu()
    L0, steps = [0, 70, 333, 700], 4
    B, T = len(L0), max(L0) + steps
    qd, kd, vd = inputs(B, Hq, Hkv, T, D, dtype, 80)
    q, k, v = to_np(qd), to_np(kd), to_np(vd)
    cache = KVCache(B, Hq, 800, D, heads_kv=Hkv, dtype=dtype, rope_base=BASE, window=window)
    if mode == "separate":
        cache.set_option(L.OPT_DECODE_FUSED, 0)
    if mode == "splits":
        cache.set_option(L.OPT_DECODE_SPLIT_ROWS, 64)
    S = max(L0)
    cache.prefill_suffix(0, None, kd[:, :, :S].contiguous(), vd[:, :, :S].contiguous(), seqlen=L0, out=False)
    cache.poison()
    if mode == "device":
        cache.set_option(L.OPT_DEVICE_LENGTHS, 1)
    idx = lambda i: torch.tensor([l + i for l in L0], device="cuda")
    row = lambda x, i: x[torch.arange(B, device="cuda"), :, idx(i)][:, :, None, :].contiguous()
    outs = [to_np(cache.append_attend(0, row(qd, i), row(kd, i), row(vd, i))) for i in range(steps)]
    cache.sync_lengths()
    Ks, Vs, Ps = storage_np(cache)
    worst = 0.0
    for b in range(B):
        n = L0[b] + steps
        ref = A.decode_steps_reference(np.transpose(q[b, :, L0[b]:n], (1, 0, 2)), k[b, :, :n], v[b, :, :n],
                                       L0[b], BASE, dtype, window=window)
        worst = max(worst, assert_close(np.stack([o[b, :, 0] for o in outs]), ref, dtype, b))
        K, V = A.stored_rows(k[b, :, :n], v[b, :, :n], np.arange(n)[None], BASE, dtype)
        np.testing.assert_array_equal(Ks[b, :, :n], K)
        np.testing.assert_array_equal(Vs[b, :, :n], V)
    assert worst <= TOL[dtype], worst
    assert cache.get_lengths(0)[0] == [l + steps for l in L0]
    cache.check()


@pytest.mark.parametrize("dtype,D,Hq,Hkv,kernel,window", [
    ("bf16", 128, 4, 2, 2, 100),      # tile kernel: the window starts inside a key tile
    ("bf16", 128, 4, 2, 2, 128),
    ("bf16", 128, 4, 4, 2, 1),
    ("bf16", 128, 2, 1, 2, 700),
    ("bf16", 128, 2, 2, 2, 5000),     # wider than every sequence: full attention
    ("bf16", 128, 4, 2, 1, 100),      # generic kernel
    ("f64", 16, 2, 2, 1, 33),
    ("bf16", 128, 4, 2, 3, 100),      # pair-of-SMs tile kernel: rank 1's first tiles lie before its window
    ("bf16", 128, 4, 4, 3, 1),
    ("bf16", 128, 2, 1, 3, 700),
    ("bf16", 128, 4, 2, 4, 100),      # persistent tile kernel
    ("bf16", 128, 32, 8, 4, 700),     # persistent, several items per CTA
    ("bf16", 128, 4, 2, 5, 100),      # two softmax threads per query row
    ("bf16", 128, 4, 4, 5, 1),
    ("bf16", 128, 2, 1, 5, 700),
])
def test_windowed_suffix_chunk_matches_full_recompute(dtype, D, Hq, Hkv, kernel, window):
    need_gpu()
    T, cuts = 1500, [1200, 37, 640]
    B = len(cuts)
    qd, kd, vd = inputs(B, Hq, Hkv, T, D, dtype, 90)
    q, k, v = to_np(qd), to_np(kd), to_np(vd)
    cache = KVCache(B, Hq, T + 20, D, heads_kv=Hkv, dtype=dtype, rope_base=BASE, window=window)
    cache.set_option(L.OPT_SUFFIX_KERNEL, kernel)
    cache.prefill_suffix(0, qd, kd, vd, out=False)
    cache.truncate(cuts)
    cache.poison()
    S = max(T - c for c in cuts)
    sel = lambda x: torch.stack([torch.nn.functional.pad(x[b, :, cuts[b]:], (0, 0, 0, S - (T - cuts[b])))
                                 for b in range(B)]).contiguous()
    got = to_np(cache.prefill_suffix(0, sel(qd), sel(kd), sel(vd), seqlen=[T - c for c in cuts]))
    for b in range(B):
        ref = A.suffix_reference(q[b, :, cuts[b]:], k[b], v[b], np.arange(T), cuts[b], BASE, dtype, window=window)
        assert_close(got[b, :, :T - cuts[b]], ref, dtype, b)
    cache.check()


CACHED = list(range(1, 9))


@pytest.mark.parametrize("seed", [7, 11, 23])
@pytest.mark.parametrize("condition,query", [
    ("window_append", CACHED + [9, 10, 11, 12]),
    ("window_edit_fifth", [1, 2, 3, 4, 20, 6, 7, 8, 9, 10, 11, 12]),
])
def test_window_cache_reuse_rule_through_library(seed, condition, query):
    """The toy decoder with a window of 4: reuse per kvc_lcp_window, then the continuation
    equals the windowed model's uncached forward."""
    need_gpu()
    E, Wl = W.toy_decoder_weights(seed)
    model = ToyDecoder(E, Wl, rope_base=BASE, window=4)
    full, _ = model.forward_full(query)
    cut = kvc.lcp(CACHED, query, window=4)
    assert cut == P.lcp_cut_window(CACHED, query, 4) == {"window_append": 8, "window_edit_fifth": 0}[condition]
    t = lambda a: torch.from_numpy(np.asarray(a)).to("cuda", torch.float64)
    Et, Wt = t(E), [tuple(t(w) for w in layer) for layer in Wl]
    cache = KVCache(1, 1, 16, 16, layers=2, dtype="f64", rope_base=BASE, window=4)

    def chunk(ids):
        h = Et[torch.as_tensor(ids, device="cuda")]
        for layer, (Wq, Wk, Wv, Wo) in enumerate(Wt):
            q, k, v = ((h @ w).reshape(1, 1, len(ids), 16).contiguous() for w in (Wq, Wk, Wv))
            a = cache.prefill_suffix(layer, q, k, v)
            h = h + torch.tanh(a.reshape(len(ids), 16) @ Wo)
        return to_np(h)

    chunk(CACHED)
    cache.truncate([cut])
    h = chunk(query[cut:])
    assert np.abs(h - full[cut:]).max() <= 1e-12
    assert cache.get_lengths(0) == ([len(query)], [len(query)])
    cache.check()
