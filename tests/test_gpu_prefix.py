"""Prefix-reuse path through libkvc: suffix-chunk parity, truncation, the
stale-position negative control, and the 2-layer toy decoder of the
prefix-reuse page driven through the library (f64, no RoPE)."""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, assert_close, device_tensor, need_gpu, storage_np, to_np
from kv_cache_append_rope_gb300 import _lib as L
from kv_cache_append_rope_gb300 import kvc
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
from oracle import attention as A
from oracle import prefix as P
from oracle.toy_decoder import ToyDecoder, sinusoidal_positions

pytestmark = pytest.mark.gpu
BASE = 10000.0


def make_inputs(B, Hq, Hkv, T, D, dtype, seed):
    qd = device_tensor(W.normal_np((B, Hq, T, D), seed), dtype)
    kd = device_tensor(W.normal_np((B, Hkv, T, D), seed + 1), dtype)
    vd = device_tensor(W.normal_np((B, Hkv, T, D), seed + 2), dtype)
    return qd, kd, vd


@pytest.mark.parametrize("dtype,D,Hq,Hkv,kernel,T,cuts", [
    ("f64", 16, 2, 2, 1, 300, [150, 0, 257]),
    ("f32", 32, 4, 2, 1, 300, [150, 0, 257]),
    ("bf16", 128, 4, 2, 1, 300, [150, 0, 257]),
    ("bf16", 128, 4, 4, 0, 300, [150, 0, 257]),      # tensor-core tile kernel (automatic)
    ("bf16", 128, 8, 2, 2, 300, [150, 0, 257]),      # tile kernel, grouped heads
    ("bf16", 128, 2, 1, 2, 1500, [1200, 37, 640]),   # tile kernel, many key tiles per query tile
    ("bf16", 128, 4, 4, 3, 300, [150, 0, 257]),      # pair-of-SMs tile kernel
    ("bf16", 128, 8, 2, 3, 300, [150, 0, 257]),
    ("bf16", 128, 2, 1, 3, 1500, [1200, 37, 640]),
    ("bf16", 128, 4, 4, 4, 300, [150, 0, 257]),      # persistent tile kernel, one item per CTA
    ("bf16", 128, 2, 1, 4, 1500, [1200, 37, 640]),
    ("bf16", 128, 32, 8, 4, 1500, [1200, 37, 640]),  # persistent: 384 items, several per CTA
    ("bf16", 128, 4, 4, 5, 300, [150, 0, 257]),      # tile kernel, two softmax threads per query row
    ("bf16", 128, 8, 2, 5, 300, [150, 0, 257]),
    ("bf16", 128, 2, 1, 5, 1500, [1200, 37, 640]),
])
def test_suffix_chunk_matches_full_recompute(dtype, D, Hq, Hkv, kernel, T, cuts):
    need_gpu()
    B, C = 3, T + 20
    qd, kd, vd = make_inputs(B, Hq, Hkv, T, D, dtype, seed=40)
    q, k, v = to_np(qd), to_np(kd), to_np(vd)
    cache = KVCache(B, Hq, C, D, heads_kv=Hkv, dtype=dtype, rope_base=BASE)
    cache.set_option(L.OPT_SUFFIX_KERNEL, kernel)
    # prefix rows, then truncate to the cuts, then the suffix chunk from position cut
    cache.prefill_suffix(0, qd, kd, vd, out=False)
    cache.truncate(cuts)
    assert cache.get_lengths(0) == (cuts, cuts)
    cache.poison()          # rows past the cuts (and past the chunk) hold keys 0, values 1e4
    S = max(T - c for c in cuts)
    sel = lambda x: torch.stack([torch.nn.functional.pad(x[b, :, cuts[b]:], (0, 0, 0, S - (T - cuts[b])))
                                 for b in range(B)]).contiguous()
    out = cache.prefill_suffix(0, sel(qd), sel(kd), sel(vd), seqlen=[T - c for c in cuts])
    got = to_np(out)
    Ks, Vs, Ps = storage_np(cache)
    for b in range(B):
        ref = A.suffix_reference(q[b, :, cuts[b]:], k[b], v[b], np.arange(T), cuts[b], BASE, dtype)
        assert_close(got[b, :, :T - cuts[b]], ref, dtype, b)
        assert np.all(got[b, :, T - cuts[b]:] == 0)            # padding rows untouched
        K, V = A.stored_rows(k[b], v[b], np.arange(T)[None], BASE, dtype)
        np.testing.assert_array_equal(Ks[b, :, :T], K)
        np.testing.assert_array_equal(Vs[b, :, :T], V)
        assert Ps[b, :T].tolist() == list(range(T))
    assert cache.get_lengths(0) == ([T] * B, [T] * B)
    cache.check()


def test_chunk_equals_repeated_decode():
    need_gpu()
    B, Hq, D, T, cut = 2, 4, 128, 96, 40
    qd, kd, vd = make_inputs(B, Hq, Hq, T, D, "bf16", seed=50)
    a = KVCache(B, Hq, T, D, dtype="bf16", rope_base=BASE)
    b = KVCache(B, Hq, T, D, dtype="bf16", rope_base=BASE)
    for c in (a, b):
        c.prefill_suffix(0, qd[:, :, :cut].contiguous(), kd[:, :, :cut].contiguous(), vd[:, :, :cut].contiguous(),
                         out=False)
    chunk = to_np(a.prefill_suffix(0, qd[:, :, cut:].contiguous(), kd[:, :, cut:].contiguous(),
                                   vd[:, :, cut:].contiguous()))
    dec = np.concatenate([to_np(b.append_attend(0, qd[:, :, i:i + 1].contiguous(), kd[:, :, i:i + 1].contiguous(),
                                                vd[:, :, i:i + 1].contiguous())) for i in range(cut, T)], axis=2)
    assert np.abs(chunk - dec).max() < 1e-2
    for x, y in zip(storage_np(a), storage_np(b)):
        np.testing.assert_array_equal(x, y)


def test_truncate_then_refill_restores_storage_and_rejects_bad_cuts():
    need_gpu()
    B, H, D, T = 2, 2, 128, 130
    qd, kd, vd = make_inputs(B, H, H, T, D, "bf16", seed=60)
    cache = KVCache(B, H, T, D, layers=2, dtype="bf16", rope_base=BASE)
    for layer in range(2):
        cache.prefill_suffix(layer, qd, kd, vd, out=False)
    full = [storage_np(cache, l) for l in range(2)]
    for bad in ([T + 1, 0], [-1, 0]):
        with pytest.raises(KVCError) as e:
            cache.truncate(bad)
        assert e.value.name == "KVC_ERR_CUT"
        assert cache.get_lengths(0) == ([T, T], [T, T])
    cache.truncate([64, 3])
    for layer in range(2):
        assert cache.get_lengths(layer) == ([64, 3], [64, 3])
        sel = lambda x: torch.stack([torch.nn.functional.pad(x[b, :, c:], (0, 0, 0, c - 3))
                                     for b, c in enumerate([64, 3])]).contiguous()
        cache.prefill_suffix(layer, sel(qd), sel(kd), sel(vd), seqlen=[T - 64, T - 3], out=False)
    for layer in range(2):
        for x, y in zip(full[layer], storage_np(cache, layer)):
            np.testing.assert_array_equal(x, y)
        assert cache.get_lengths(layer) == ([T, T], [T, T])
    cache.check()


def test_stale_next_position_negative_control():
    need_gpu()
    B, H, D, T, cut, old = 1, 2, 16, 12, 4, 8
    qd, kd, vd = make_inputs(B, H, H, T, D, "f64", seed=70)
    q, k, v = to_np(qd), to_np(kd), to_np(vd)
    results = {}
    for name, start in (("correct", None), ("stale", [old])):
        cache = KVCache(B, H, 32, D, dtype="f64", rope_base=BASE)
        cache.prefill_suffix(0, qd[:, :, :old].contiguous(), kd[:, :, :old].contiguous(),
                             vd[:, :, :old].contiguous(), out=False)
        cache.truncate([cut])
        out = cache.prefill_suffix(0, qd[:, :, cut:].contiguous(), kd[:, :, cut:].contiguous(),
                                   vd[:, :, cut:].contiguous(), start_pos=start)
        results[name] = to_np(out)[0]
        assert cache.get_lengths(0) == ([T], [T if start is None else old + T - cut])
        assert storage_np(cache)[2][0, :T].tolist() == (list(range(T)) if start is None else
                                                        list(range(cut)) + list(range(old, old + T - cut)))
    good = A.suffix_reference(q[0, :, cut:], k[0], v[0], np.arange(T), cut, BASE, "f64")
    stale_pos = np.concatenate([np.arange(cut), old + np.arange(T - cut)])
    stale = A.suffix_reference(q[0, :, cut:], k[0], v[0], stale_pos, cut, BASE, "f64")
    assert np.abs(results["correct"] - good).max() <= 1e-12
    assert np.abs(results["stale"] - stale).max() <= 1e-12
    assert np.abs(results["stale"] - good).max() > 1e-12


# ---- the prefix-reuse page's 2-layer decoder, attention through libkvc -------------

def _pe_torch(positions, d):
    """The oracle's additive sinusoid (pinned by tests/test_oracle_sinusoid.py), on the GPU."""
    return torch.from_numpy(sinusoidal_positions(positions, d)).to("cuda")


class GpuToyDecoder:
    """Embedding, projections and tanh residual in torch; attention and cache in libkvc."""

    def __init__(self, E, Wl):
        t = lambda a: torch.from_numpy(np.asarray(a)).to("cuda", torch.float64)
        self.E = t(E)
        self.W = [tuple(t(w) for w in layer) for layer in Wl]
        self.d = self.E.shape[1]
        self.cache = KVCache(1, 1, 16, self.d, layers=len(self.W), dtype="f64", rope_base=0.0)
        self.projected_rows = 0

    def chunk(self, ids, start=None):
        _, nxt = self.cache.get_lengths(0)
        p0 = nxt[0] if start is None else start
        h = self.E[torch.as_tensor(ids, device="cuda")] + _pe_torch(np.arange(p0, p0 + len(ids)), self.d)
        for layer, (Wq, Wk, Wv, Wo) in enumerate(self.W):
            q, k, v = (h @ w for w in (Wq, Wk, Wv))
            self.projected_rows += 3 * len(ids)
            shape = (1, 1, len(ids), self.d)
            a = self.cache.prefill_suffix(layer, q.reshape(shape).contiguous(), k.reshape(shape).contiguous(),
                                          v.reshape(shape).contiguous(),
                                          start_pos=None if start is None else [start])
            h = h + torch.tanh(a.reshape(len(ids), self.d) @ Wo)
        return to_np(h)


CONDITIONS = {
    "append": (list(range(1, 9)), list(range(1, 13))),
    "edit_first": (list(range(1, 9)), [20] + list(range(2, 13))),
    "edit_fifth": (list(range(1, 9)), [1, 2, 3, 4, 20, 6, 7, 8, 9, 10, 11, 12]),
    "edit_eighth": (list(range(1, 9)), list(range(1, 8)) + [20, 9, 10, 11, 12]),
    "shortened": (list(range(1, 9)), [1, 2, 3, 4]),
    "branch_append": ([1, 2, 3, 4, 5, 20, 21, 22], [1, 2, 3, 4, 5, 20, 21, 22, 9, 10, 11, 12]),
    "full_hit": (list(range(1, 9)), list(range(1, 9))),
}


@pytest.mark.parametrize("seed", [7, 11, 23])
@pytest.mark.parametrize("condition", list(CONDITIONS))
def test_toy_decoder_prefix_reuse_through_library(seed, condition):
    need_gpu()
    cached, query = CONDITIONS[condition]
    E, Wl = W.toy_decoder_weights(seed)
    oracle_model = ToyDecoder(E, Wl)
    full_h, _ = oracle_model.forward_full(query)
    for stale in (False, True):
        gpu = GpuToyDecoder(E, Wl)
        gpu.chunk(cached)
        cut = kvc.lcp(cached, query)
        assert cut == P.lcp_cut(cached, query)
        gpu.cache.truncate([cut])
        gpu.projected_rows = 0
        h = gpu.chunk(query[cut:], start=len(cached) if stale else None)
        assert gpu.projected_rows == P.projection_rows(2, len(query), cut)
        err = np.abs(h - full_h[cut:]).max()
        if not stale:
            assert err <= 1e-12
        elif cut == len(cached):
            assert err <= 1e-12                       # plain append: nothing is stale
        else:
            assert err > 1e-12
        gpu.cache.check()


@pytest.mark.parametrize("window", [0, 300])
def test_persistent_tile_kernel_equals_the_one_item_kernel(window):
    """The persistent tile kernel (one CTA per SM walking the work list, barriers counting
    across items, the next item's loads and QK^T overlapping the epilogue) computes every
    item as the one-item-per-CTA kernel does: outputs equal bit for bit, with several items
    per CTA, ragged sequences and a sliding window."""
    need_gpu()
    B, Hq, Hkv, D, T = 4, 32, 8, 128, 1400
    cuts = [1100, 0, 613, 1333]
    qd, kd, vd = make_inputs(B, Hq, Hkv, T, D, "bf16", seed=45)
    S = max(T - c for c in cuts)
    sel = lambda x: torch.stack([torch.nn.functional.pad(x[b, :, cuts[b]:], (0, 0, 0, S - (T - cuts[b])))
                                 for b in range(B)]).contiguous()
    outs = []
    for kernel in (2, 4):
        cache = KVCache(B, Hq, T + 20, D, heads_kv=Hkv, dtype="bf16", rope_base=BASE, window=window)
        cache.set_option(L.OPT_SUFFIX_KERNEL, kernel)
        cache.prefill_suffix(0, qd, kd, vd, out=False)
        cache.truncate(cuts)
        cache.poison()
        outs.append(to_np(cache.prefill_suffix(0, sel(qd), sel(kd), sel(vd), seqlen=[T - c for c in cuts])))
        assert cache.kernel_stats("suffix")[1] == 1
        cache.check()
    np.testing.assert_array_equal(outs[0], outs[1])
