"""Device-length decode steps, CUDA-graph replay and bf16 outputs, against the oracle.

With KVC_OPT_DEVICE_LENGTHS the decode kernel reads each sequence's length and
next position from device memory, so one captured step can be replayed while the
cache grows.  Each replayed step must equal the float64 oracle's full-prefix
recomputation ([Ch37] listing "Evaluate one newest query across the retained
rows plus the candidate key/value row before committing the append") within the
bf16 tolerance, and the stored rows, positions and lengths must be bit-exact.
A step in which one sequence is full is rejected as a whole ([Ch37] "Reset or
reject without corrupting retained state"), here on the device.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, device_tensor, need_gpu, raw_storage_np, storage_np, to_np
from kv_cache_append_rope_gb300 import _lib as L
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
from oracle import attention as A

pytestmark = pytest.mark.gpu
BASE = 10000.0


def inputs(B, Hq, Hkv, T, seed):
    q = device_tensor(W.normal_np((B, Hq, T, 128), seed), "bf16")
    k = device_tensor(W.normal_np((B, Hkv, T, 128), seed + 1), "bf16")
    v = device_tensor(W.normal_np((B, Hkv, T, 128), seed + 2), "bf16")
    return q, k, v


def prefilled(L0, Hq, Hkv, C, qkv):
    q, k, v = qkv
    cache = KVCache(len(L0), Hq, C, 128, heads_kv=Hkv, rope_base=BASE)
    S = max(max(L0), 1)
    cache.prefill_suffix(0, None, k[:, :, :S].contiguous(), v[:, :, :S].contiguous(), seqlen=L0, out=False)
    return cache


def step_rows(x, L0, i):
    """Row L0[b] + i of every sequence, as a [B, H, 1, d] tensor."""
    idx = torch.tensor([l + i for l in L0], device="cuda")
    return x[torch.arange(len(L0), device="cuda"), :, idx][:, :, None, :].contiguous()


def check_steps(cache, outs, qkv, L0, steps):
    q, k, v = (to_np(x) for x in qkv)
    Ks, Vs, Ps = storage_np(cache)
    worst = 0.0
    for b in range(len(L0)):
        n = L0[b] + steps
        ref = A.decode_steps_reference(np.transpose(q[b, :, L0[b]:n], (1, 0, 2)), k[b, :, :n], v[b, :, :n],
                                       L0[b], BASE, "bf16")
        got = np.stack([o[b, :, 0] for o in outs])
        worst = max(worst, np.abs(got - ref).max())
        K, V = A.stored_rows(k[b, :, :n], v[b, :, :n], np.arange(n)[None], BASE, "bf16")
        np.testing.assert_array_equal(Ks[b, :, :n], K)
        np.testing.assert_array_equal(Vs[b, :, :n], V)
        assert Ps[b, :n].tolist() == list(range(n))
    assert worst <= TOL["bf16"], worst


@pytest.mark.parametrize("Hq,Hkv,L0,split_rows", [
    (8, 2, [0, 70, 333, 700], 0),       # G = 4: one launch per step, in-kernel merge
    (8, 2, [5, 333, 700], 128),         # several splits per sequence
    (32, 1, [1, 100, 257, 63], 0),      # MQA: decode + merge launches
])
def test_device_lengths_match_oracle(Hq, Hkv, L0, split_rows):
    need_gpu()
    steps = 4
    qkv = inputs(len(L0), Hq, Hkv, max(L0) + steps, 7)
    cache = prefilled(L0, Hq, Hkv, 800, qkv)
    if split_rows:
        cache.set_option(L.OPT_DECODE_SPLIT_ROWS, split_rows)
    cache.set_option(L.OPT_DEVICE_LENGTHS, 1)
    q, k, v = qkv
    outs = [to_np(cache.append_attend(0, step_rows(q, L0, i), step_rows(k, L0, i), step_rows(v, L0, i)))
            for i in range(steps)]
    cache.sync_lengths()
    lens, nexts = cache.get_lengths(0)
    assert lens == [l + steps for l in L0] and nexts == lens
    check_steps(cache, outs, qkv, L0, steps)
    cache.check()


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (32, 1)])
def test_graph_replay_grows_the_cache(Hq, Hkv):
    """One captured decode step replayed N times: N correct steps, lengths advanced on the device."""
    need_gpu()
    L0, replays = [3, 120, 64, 500, 257], 6
    steps = 1 + replays
    qkv = inputs(len(L0), Hq, Hkv, max(L0) + steps, 11)
    q, k, v = qkv
    cache = prefilled(L0, Hq, Hkv, 1024, qkv)
    cache.set_option(L.OPT_DEVICE_LENGTHS, 1)
    qs, ks, vs = step_rows(q, L0, 0), step_rows(k, L0, 0), step_rows(v, L0, 0)
    out = torch.empty(qs.shape, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        cache.append_attend(0, qs, ks, vs, out=out)            # uncaptured step 0 (allocates split scratch)
    torch.cuda.current_stream().wait_stream(side)
    outs = [to_np(out)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cache.append_attend(0, qs, ks, vs, out=out)            # recorded, not run
    for i in range(1, steps):
        qs.copy_(step_rows(q, L0, i))
        ks.copy_(step_rows(k, L0, i))
        vs.copy_(step_rows(v, L0, i))
        g.replay()
        outs.append(to_np(out))
    cache.sync_lengths()
    lens, nexts = cache.get_lengths(0)
    assert lens == [l + steps for l in L0] and nexts == lens
    check_steps(cache, outs, qkv, L0, steps)
    cache.check()
    del g


def test_device_full_rejects_the_whole_step():
    need_gpu()
    L0, C = [10, 127, 50], 128
    qkv = inputs(3, 4, 4, 130, 21)
    q, k, v = qkv
    cache = prefilled(L0, 4, 4, C, qkv)
    cache.set_option(L.OPT_DEVICE_LENGTHS, 1)
    cache.append_attend(0, step_rows(q, L0, 0), step_rows(k, L0, 0), step_rows(v, L0, 0))   # fills sequence 1
    cache.check()
    K0, V0, P0 = raw_storage_np(cache)
    cache.append_attend(0, step_rows(q, L0, 1), step_rows(k, L0, 1), step_rows(v, L0, 1))   # rejected on the device
    with pytest.raises(KVCError) as e:
        cache.check()
    assert e.value.name == "KVC_ERR_DEVICE" and "cache full" in str(e.value)
    cache.sync_lengths()
    assert cache.get_lengths(0) == ([11, 128, 51], [11, 128, 51])
    K1, V1, P1 = raw_storage_np(cache)
    np.testing.assert_array_equal(K0, K1)
    np.testing.assert_array_equal(V0, V1)
    np.testing.assert_array_equal(P0, P1)


@pytest.mark.parametrize("Hq,Hkv,split_rows,fused", [
    (8, 2, 0, True), (8, 2, 128, True), (32, 1, 0, True), (8, 2, 128, False)])
def test_bf16_output_is_the_rounded_float32_output(Hq, Hkv, split_rows, fused):
    need_gpu()
    L0, steps = [5, 333, 700], 3
    qkv = inputs(len(L0), Hq, Hkv, max(L0) + steps, 31)
    q, k, v = qkv
    caches = [prefilled(L0, Hq, Hkv, 800, qkv) for _ in range(2)]
    for c in caches:
        if split_rows:
            c.set_option(L.OPT_DECODE_SPLIT_ROWS, split_rows)
        if not fused:
            c.set_option(L.OPT_DECODE_FUSED, 0)
    for i in range(steps):
        args = (step_rows(q, L0, i), step_rows(k, L0, i), step_rows(v, L0, i))
        o32 = caches[0].append_attend(0, *args)
        o16 = caches[1].append_attend(0, *args, out=torch.empty(o32.shape, dtype=torch.bfloat16, device="cuda"))
        assert torch.equal(o16, o32.to(torch.bfloat16))
    for c in caches:
        c.check()


def test_bf16_output_needs_bf16_storage():
    need_gpu()
    cache = KVCache(1, 4, 64, 128, dtype="f32", rope_base=BASE)
    x = torch.zeros((1, 4, 1, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(KVCError) as e:
        cache.append_attend(0, x, x, x, out=torch.zeros((1, 4, 1, 128), dtype=torch.bfloat16, device="cuda"))
    assert e.value.name == "KVC_ERR_DTYPE"
    assert cache.get_lengths(0) == ([0], [0])


def test_device_checked_truncate():
    need_gpu()
    L0 = [10, 40, 25]
    qkv = inputs(3, 4, 4, 41, 41)
    cache = prefilled(L0, 4, 4, 64, qkv)
    cache.set_option(L.OPT_DEVICE_LENGTHS, 1)
    cache.truncate([5, 41, 0])                 # 41 > 40: rejected on the device, nothing changes
    with pytest.raises(KVCError) as e:
        cache.check()
    assert e.value.name == "KVC_ERR_DEVICE" and "cut beyond" in str(e.value)
    cache.sync_lengths()
    assert cache.get_lengths(0) == (L0, L0)
    fresh = prefilled(L0, 4, 4, 64, qkv)
    fresh.set_option(L.OPT_DEVICE_LENGTHS, 1)
    fresh.truncate([5, 40, 0])
    fresh.check()
    assert fresh.get_lengths(0) == ([5, 40, 0], [5, 40, 0])
