"""Model-wide decode sessions: prepare one step per layer, then commit them together.

[Ch37] listing "Evaluate one newest query across the retained rows plus the
candidate key/value row before committing the append": a prepared step carries
its candidate rows and the cache length it expects, and (as the listing's comment
announces for chapter 38) a model prepares one such ticket per decoder block,
finishes the model, checks that every ticket still targets its cache, and only
then commits the complete stack.  Here kvc_prepare_attend stages the candidate
rows beyond the logical length and kvc_commit advances every named layer at once
or none of them.

The model is the [LCP5] two-layer toy decoder with rotary positions (the
oracle's ToyDecoder with rope_base): prefill of ragged prompts, then greedy
one-token decode steps through the tied vocabulary head, every hidden state
against the oracle's uncached forward within 1e-12 (float64 storage).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import device_tensor, need_gpu, storage_np, to_np
from kv_cache_append_rope_gb300 import _lib as L
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
from oracle.toy_decoder import ToyDecoder

pytestmark = pytest.mark.gpu
BASE = 10000.0


class GpuRopeDecoder:
    """Embedding, projections, residual and vocabulary head in torch; attention and cache in libkvc."""

    def __init__(self, E, Wl, B, C):
        t = lambda a: torch.from_numpy(np.asarray(a)).to("cuda", torch.float64)
        self.E = t(E)
        self.W = [tuple(t(w) for w in layer) for layer in Wl]
        self.d = self.E.shape[1]
        self.B = B
        self.cache = KVCache(B, 1, C, self.d, layers=len(self.W), dtype="f64", rope_base=BASE)

    def prefill(self, prompts):
        S = max(len(p) for p in prompts)
        ids = torch.zeros((self.B, S), dtype=torch.long, device="cuda")
        for b, p in enumerate(prompts):
            ids[b, :len(p)] = torch.tensor(p, device="cuda")
        h = self.E[ids]                                          # [B, S, d]
        for layer, (Wq, Wk, Wv, Wo) in enumerate(self.W):
            q, k, v = ((h @ w)[:, None].contiguous() for w in (Wq, Wk, Wv))
            a = self.cache.prefill_suffix(layer, q, k, v, seqlen=[len(p) for p in prompts])
            h = h + torch.tanh(a[:, 0] @ Wo)
        return [to_np(h[b, :len(p)]) for b, p in enumerate(prompts)]

    def decode(self, ids, commit=True):
        """One token per sequence through every layer (prepared), then one commit."""
        h = self.E[torch.as_tensor(ids, device="cuda")]              # [B, d]
        tickets = []
        for layer, (Wq, Wk, Wv, Wo) in enumerate(self.W):
            q, k, v = ((h @ w)[:, None, None].contiguous() for w in (Wq, Wk, Wv))
            a, ticket = self.cache.prepare_attend(layer, q, k, v)
            tickets.append(ticket)
            h = h + torch.tanh(a[:, 0, 0] @ Wo)
        if commit:
            self.cache.commit(tickets)
        return to_np(h), tickets

    def greedy(self, h_rows):
        return [int(np.argmax(r @ to_np(self.E).T)) for r in h_rows]


@pytest.mark.parametrize("seed", [7, 11, 23])
def test_session_generation_matches_uncached_oracle(seed):
    need_gpu()
    E, Wl = W.toy_decoder_weights(seed)
    rng = np.random.default_rng(seed)
    prompts = [rng.integers(0, 32, size=5).tolist(), rng.integers(0, 32, size=9).tolist()]
    gpu = GpuRopeDecoder(E, Wl, B=2, C=32)
    h_prompt = gpu.prefill(prompts)
    seqs = [list(p) for p in prompts]
    hidden = [list(h) for h in h_prompt]
    nxt = gpu.greedy([h[-1] for h in h_prompt])
    for _ in range(4):
        for b in range(2):
            seqs[b].append(nxt[b])
        h, _ = gpu.decode(nxt)
        for b in range(2):
            hidden[b].append(h[b])
        nxt = gpu.greedy(h)
    model = ToyDecoder(E, Wl, rope_base=BASE)
    for b in range(2):
        ref, _ = model.forward_full(seqs[b])
        assert np.abs(np.stack(hidden[b]) - ref).max() <= 1e-12
        # the oracle picks the same greedy tokens unless two logits are within 1e-9
        logits = model.logits(ref[len(prompts[b]) - 1:-1])
        for row, chosen in zip(logits, seqs[b][len(prompts[b]):]):
            top2 = np.sort(row)[-2:]
            if top2[1] - top2[0] > 1e-9:
                assert int(np.argmax(row)) == chosen
    lens, nexts = gpu.cache.get_lengths(1)
    assert lens == [len(s) for s in seqs] and nexts == lens
    gpu.cache.check()


def test_prepared_steps_commit_all_or_nothing():
    need_gpu()
    E, Wl = W.toy_decoder_weights(7)
    gpu = GpuRopeDecoder(E, Wl, B=2, C=32)
    gpu.prefill([[1, 2, 3], [4, 5, 6, 7]])
    lengths = lambda: [gpu.cache.get_lengths(l)[0] for l in range(2)]
    assert lengths() == [[3, 4], [3, 4]]
    # prepared, not committed: lengths unchanged
    _, tickets = gpu.decode([8, 9], commit=False)
    assert lengths() == [[3, 4], [3, 4]]
    # a repeated layer, a foreign ticket: rejected, nothing committed
    for bad in ([tickets[0], tickets[0]], [tickets[0], GpuRopeDecoder(E, Wl, 2, 32).decode([1, 1], False)[1][1]]):
        with pytest.raises(KVCError) as e:
            gpu.cache.commit(bad)
        assert e.value.name == "KVC_ERR_TICKET"
        assert lengths() == [[3, 4], [3, 4]]
    gpu.cache.commit([])                                          # nothing to commit
    gpu.cache.commit(tickets)
    assert lengths() == [[4, 5], [4, 5]]
    # committed tickets cannot commit again (the layers changed)
    with pytest.raises(KVCError):
        gpu.cache.commit(tickets)
    # a truncate between prepare and commit makes the tickets stale
    _, tickets = gpu.decode([10, 11], commit=False)
    gpu.cache.truncate([2, 2])
    with pytest.raises(KVCError) as e:
        gpu.cache.commit(tickets)
    assert e.value.name == "KVC_ERR_TICKET" and "stale" in str(e.value)
    assert lengths() == [[2, 2], [2, 2]]
    gpu.cache.check()


def test_reprepared_layer_invalidates_the_earlier_ticket():
    need_gpu()
    E, Wl = W.toy_decoder_weights(11)
    prompts = [[1, 2, 3, 4], [5, 6]]
    gpu = GpuRopeDecoder(E, Wl, B=2, C=32)
    gpu.prefill(prompts)
    _, first = gpu.decode([7, 8], commit=False)
    h, second = gpu.decode([9, 10], commit=False)                 # same slots, new candidate rows
    with pytest.raises(KVCError):
        gpu.cache.commit(first)
    gpu.cache.commit(second)
    model = ToyDecoder(E, Wl, rope_base=BASE)
    for b, tok in enumerate([9, 10]):
        ref, _ = model.forward_full(prompts[b] + [tok])
        assert np.abs(h[b] - ref[-1]).max() <= 1e-12
    gpu.cache.check()


@pytest.mark.parametrize("Hq,Hkv,fused", [(8, 2, True), (32, 1, True), (8, 2, False)])
def test_prepare_then_commit_equals_append(Hq, Hkv, fused):
    """bf16 tensor-core path: prepare + commit gives the outputs and storage of append_attend."""
    need_gpu()
    L0, steps, layers = [5, 300, 129], 3, 2
    B, T = len(L0), max(L0) + steps
    kv = [device_tensor(W.normal_np((B, Hkv, T, 128), 50 + i), "bf16") for i in range(2 * layers)]
    qs = [device_tensor(W.normal_np((B, Hq, T, 128), 60 + l), "bf16") for l in range(layers)]
    caches = []
    for _ in range(2):
        c = KVCache(B, Hq, 512, 128, heads_kv=Hkv, layers=layers, rope_base=BASE)
        if not fused:
            c.set_option(L.OPT_DECODE_FUSED, 0)
        for l in range(layers):
            c.prefill_suffix(l, None, kv[2 * l][:, :, :max(L0)].contiguous(),
                             kv[2 * l + 1][:, :, :max(L0)].contiguous(), seqlen=L0, out=False)
        caches.append(c)
    idx = lambda i: torch.tensor([l + i for l in L0], device="cuda")
    row = lambda x, i: x[torch.arange(B, device="cuda"), :, idx(i)][:, :, None, :].contiguous()
    for i in range(steps):
        tickets = []
        for l in range(layers):
            a = caches[0].append_attend(l, row(qs[l], i), row(kv[2 * l], i), row(kv[2 * l + 1], i))
            p, t = caches[1].prepare_attend(l, row(qs[l], i), row(kv[2 * l], i), row(kv[2 * l + 1], i))
            tickets.append(t)
            assert torch.equal(a, p)
        caches[1].commit(tickets)
    for l in range(layers):
        assert caches[0].get_lengths(l) == caches[1].get_lengths(l)
        for x, y in zip(storage_np(caches[0], l), storage_np(caches[1], l)):
            np.testing.assert_array_equal(x, y)
    for c in caches:
        c.check()


def test_prepare_is_refused_with_device_lengths():
    need_gpu()
    c = KVCache(1, 4, 64, 128, rope_base=BASE)
    c.set_option(L.OPT_DEVICE_LENGTHS, 1)
    x = torch.zeros((1, 4, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(KVCError) as e:
        c.prepare_attend(0, x, x, x)
    assert e.value.name == "KVC_ERR_CONFIG"
