"""Decode-step parity of libkvc against the float64 oracle.

Every call goes through the C ABI (kv_cache_append_rope_gb300.kvc).  Inputs are
seeded; the oracle sees exactly the storage-dtype values the GPU sees.
Tolerances: f64 1e-12, f32 1e-5, bf16 2e-2 (max abs); stored rows, positions and
lengths bit-exact.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, assert_close, device_tensor, need_gpu, storage_np, to_np
from kv_cache_append_rope_gb300 import _lib as L
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache
from oracle import attention as A

pytestmark = pytest.mark.gpu
BASE = 10000.0


def run_decode(dtype, D, Hq, Hkv, L0, steps, C, generic=False, split_rows=0, seed=0, fused=True, tc=True,
               window=0, out_dtype=None, lanes=True, block_rows=0, streamk=True):
    """Prefill ragged prefixes, run `steps` decode steps; return (cache, outs, inputs)."""
    need_gpu()
    B = len(L0)
    T = max(L0) + steps
    q = W.normal_np((B, Hq, T, D), seed)
    k = W.normal_np((B, Hkv, T, D), seed + 1)
    v = W.normal_np((B, Hkv, T, D), seed + 2)
    qd, kd, vd = (device_tensor(x, dtype) for x in (q, k, v))
    q, k, v = to_np(qd), to_np(kd), to_np(vd)        # the exact values the GPU sees
    cache = KVCache(B, Hq, C, D, heads_kv=Hkv, dtype=dtype, rope_base=BASE, window=window, block_rows=block_rows)
    if not tc:
        cache.set_option(L.OPT_DECODE_TC, 0)
    if not lanes:
        cache.set_option(L.OPT_DECODE_LANES, 0)
    if not streamk:
        cache.set_option(L.OPT_DECODE_STREAMK, 0)
    if generic:
        cache.set_option(L.OPT_FORCE_GENERIC, 1)
    if split_rows:
        cache.set_option(L.OPT_DECODE_SPLIT_ROWS, split_rows)
    if not fused:
        cache.set_option(L.OPT_DECODE_FUSED, 0)
    S = max(max(L0), 1)
    cache.prefill_suffix(0, qd[:, :, :S].contiguous(), kd[:, :, :S].contiguous(), vd[:, :, :S].contiguous(),
                         seqlen=L0, out=False)
    cache.poison()          # rows past every length: keys 0, values 1e4 -- a leaked row shows
    outs = []
    for i in range(steps):
        idx = torch.tensor([l + i for l in L0], device="cuda")
        sel = lambda x: x[torch.arange(B, device="cuda"), :, idx][:, :, None, :].contiguous()
        out = None if out_dtype is None else torch.empty((B, Hq, 1, D), dtype=out_dtype, device="cuda")
        outs.append(to_np(cache.append_attend(0, sel(qd), sel(kd), sel(vd), out=out)))
    torch.cuda.synchronize()
    return cache, outs, (q, k, v)


def check_against_oracle(dtype, cache, outs, qkv, L0, steps, window=0):
    q, k, v = qkv
    B = len(L0)
    worst = 0.0
    Ks, Vs, Ps = storage_np(cache)
    for b in range(B):
        n = L0[b] + steps
        ref = A.decode_steps_reference(np.transpose(q[b, :, L0[b]:n], (1, 0, 2)), k[b, :, :n], v[b, :, :n],
                                       L0[b], BASE, dtype, window=window)
        got = np.stack([o[b, :, 0] for o in outs])
        worst = max(worst, assert_close(got, ref, dtype, b))
        K, V = A.stored_rows(k[b, :, :n], v[b, :, :n], np.arange(n)[None], BASE, dtype)
        np.testing.assert_array_equal(Ks[b, :, :n], K)          # rotated, rounded keys: bit-exact
        np.testing.assert_array_equal(Vs[b, :, :n], V)
        assert Ps[b, :n].tolist() == list(range(n))
    assert worst <= TOL[dtype], worst
    lens, nexts = cache.get_lengths(0)
    assert lens == [l + steps for l in L0] and nexts == lens
    cache.check()
    return worst


@pytest.mark.parametrize("dtype,D,Hq,Hkv,generic", [
    ("f64", 16, 4, 2, True),
    ("f32", 64, 4, 4, True),
    ("bf16", 64, 4, 1, True),
    ("bf16", 128, 4, 4, True),
    ("bf16", 128, 4, 4, False),
    ("bf16", 128, 8, 2, False),
])
def test_decode_matches_oracle(dtype, D, Hq, Hkv, generic):
    L0, steps = [0, 70, 200], 5
    cache, outs, qkv = run_decode(dtype, D, Hq, Hkv, L0, steps, C=300, generic=generic)
    check_against_oracle(dtype, cache, outs, qkv, L0, steps)


@pytest.mark.parametrize("Hkv", [8, 1])
def test_gqa_mqa_fast_path(Hkv):
    L0, steps = [1, 100, 257, 63], 3
    cache, outs, qkv = run_decode("bf16", 128, 32, Hkv, L0, steps, C=400)
    check_against_oracle("bf16", cache, outs, qkv, L0, steps)


@pytest.mark.parametrize("Hq,Hkv,split_rows,window", [
    (32, 1, 0, 0), (32, 1, 128, 0), (32, 1, 1024, 0), (32, 2, 0, 300), (48, 2, 256, 0), (32, 1, 64, 100),
])
def test_tensor_core_decode_matches_oracle_and_the_mma_sync_path(Hq, Hkv, split_rows, window):
    """16 < G <= 32 query heads per key/value head run on the tcgen05 decode kernel: the
    oracle, the m16n8k16 kernel (KVC_OPT_DECODE_TC = 0) and bf16 outputs agree."""
    L0, steps = [1, 100, 257, 700], 3
    cache, outs, qkv = run_decode("bf16", 128, Hq, Hkv, L0, steps, C=800, split_rows=split_rows, window=window)
    check_against_oracle("bf16", cache, outs, qkv, L0, steps, window=window)
    _, ref, _ = run_decode("bf16", 128, Hq, Hkv, L0, steps, C=800, split_rows=split_rows, window=window, tc=False)
    assert np.abs(np.stack(outs) - np.stack(ref)).max() < 1e-2
    _, o16, _ = run_decode("bf16", 128, Hq, Hkv, L0, steps, C=800, split_rows=split_rows, window=window,
                           out_dtype=torch.bfloat16)
    np.testing.assert_array_equal(np.stack(o16), to_np(torch.from_numpy(np.stack(outs)).to(torch.bfloat16)))


@pytest.mark.parametrize("Hq,Hkv,window,B", [(32, 1, 0, 64), (32, 2, 0, 40), (24, 1, 0, 64), (32, 1, 200, 64),
                                              (32, 1, 0, 256)])   # 256 lanes: the plan's limit
def test_streamk_tensor_core_decode_matches_oracle(Hq, Hkv, window, B):
    """Stream-K tensor-core decode (KVC_OPT_DECODE_STREAMK, the default): the lanes' 128-key
    tiles laid end to end and cut into one equal run per SM, so that with these short ragged
    lanes most CTAs span two or three lanes and most lanes several CTAs.  Every sequence
    against the oracle (stored rows bit for bit, lengths), and the outputs against the
    per-sequence piece plan."""
    rng = np.random.default_rng(B + Hq + window)
    L0 = rng.integers(0, 700, size=B).tolist()
    L0[:6] = [0, 1, 127, 128, 255, 699]
    steps = 2
    cache, outs, qkv = run_decode("bf16", 128, Hq, Hkv, L0, steps, C=704, window=window, seed=5)
    check_against_oracle("bf16", cache, outs, qkv, L0, steps, window=window)
    _, ref, _ = run_decode("bf16", 128, Hq, Hkv, L0, steps, C=704, window=window, seed=5, streamk=False)
    assert np.abs(np.stack(outs) - np.stack(ref)).max() < 1e-2


@pytest.mark.parametrize("Hq,Hkv,window,block_rows,out_bf16,B", [
    (32, 32, 0, 0, False, 48), (32, 8, 0, 0, False, 160), (32, 32, 100, 0, False, 48), (32, 32, 0, 64, False, 48),
    (32, 32, 0, 0, True, 48), (32, 32, 0, 0, False, 58),
])
def test_many_short_lanes_per_cta_match_oracle(Hq, Hkv, window, block_rows, out_bf16, B):
    """Short ragged contexts with many lanes run on CTAs that walk several lanes each
    (KVC_OPT_DECODE_LANES): every sampled sequence against the oracle, stored rows bit
    for bit, and the outputs against the one-CTA-per-lane path.  At least four waves of
    lanes; on 152 SMs B = 48 gives 6 lanes per CTA in whole CTAs, B = 58 gives 7 lanes
    per CTA with one lane in the last CTA."""
    L0 = np.random.default_rng(B + Hkv).integers(0, 301, size=B).tolist()
    L0[0], L0[1] = 0, 300
    steps = 3
    od = torch.bfloat16 if out_bf16 else None
    cache, outs, qkv = run_decode("bf16", 128, Hq, Hkv, L0, steps, C=320, window=window, block_rows=block_rows,
                                  out_dtype=od, seed=7)
    q, k, v = qkv
    Ks, Vs, Ps = storage_np(cache)
    got = np.stack(outs)
    for b in sorted(set([0, 1] + list(range(2, B, max(1, B // 10))))):
        n = L0[b] + steps
        ref = A.decode_steps_reference(np.transpose(q[b, :, L0[b]:n], (1, 0, 2)), k[b, :, :n], v[b, :, :n],
                                       L0[b], BASE, "bf16", window=window)
        if out_bf16:
            assert np.abs(got[:, b, :, 0] - ref).max() <= TOL["bf16"]
        else:
            assert_close(got[:, b, :, 0], ref, "bf16", b)
        K, V = A.stored_rows(k[b, :, :n], v[b, :, :n], np.arange(n)[None], BASE, "bf16")
        np.testing.assert_array_equal(Ks[b, :, :n], K)
        np.testing.assert_array_equal(Vs[b, :, :n], V)
        assert Ps[b, :n].tolist() == list(range(n))
    assert cache.get_lengths(0)[0] == [l + steps for l in L0]
    cache.check()
    _, ref_outs, _ = run_decode("bf16", 128, Hq, Hkv, L0, steps, C=320, window=window, block_rows=block_rows,
                                out_dtype=od, seed=7, lanes=False)
    assert np.abs(got - np.stack(ref_outs)).max() < 1e-2


def test_split_sizes_agree():
    """One split, two, several and one per 64 rows: same outputs (log-sum-exp merge)."""
    L0, steps = [5, 333, 700], 2
    results = []
    for rows in [1024, 448, 128, 64, 0]:
        cache, outs, qkv = run_decode("bf16", 128, 8, 2, L0, steps, C=800, split_rows=rows)
        check_against_oracle("bf16", cache, outs, qkv, L0, steps)
        results.append(np.stack(outs))
    for r in results[1:]:
        assert np.abs(r - results[0]).max() < 5e-3


def test_generic_and_fast_paths_agree():
    L0, steps = [3, 150], 3
    _, a, _ = run_decode("bf16", 128, 4, 4, L0, steps, C=200, generic=True)
    _, b, _ = run_decode("bf16", 128, 4, 4, L0, steps, C=200, generic=False)
    assert np.abs(np.stack(a) - np.stack(b)).max() < 1e-2


def test_first_step_returns_the_value():
    """t = 1: the single weight is 1 and the output is the (rounded) new value row."""
    cache, outs, (q, k, v) = run_decode("bf16", 128, 4, 4, [0], 1, C=8)
    np.testing.assert_allclose(outs[0][0, :, 0], v[0, :, 0], atol=1e-6)


def test_appended_keys_bit_exact_at_volume():
    """Millions of appended bf16 key elements, at small and large positions, equal the
    oracle's float64 rotation rounded to bf16 bit for bit (this exercises the rare
    elements whose float32 rotation lands next to a bf16 rounding boundary)."""
    need_gpu()
    B, H, T, D = 2, 8, 4096, 128
    start = [0, 28000]
    kd = device_tensor(W.normal_np((B, H, T, D), 81), "bf16")
    vd = device_tensor(W.normal_np((B, H, T, D), 82), "bf16")
    cache = KVCache(B, H, T, D, dtype="bf16", rope_base=BASE, rope_max_positions=32768)
    cache.prefill_suffix(0, None, kd, vd, start_pos=start, out=False)
    Ks, Vs, Ps = storage_np(cache)
    k, v = to_np(kd), to_np(vd)
    for b in range(B):
        pos = start[b] + np.arange(T)
        K, V = A.stored_rows(k[b], v[b], pos[None, :], BASE, "bf16")
        np.testing.assert_array_equal(Ks[b], K)
        np.testing.assert_array_equal(Vs[b], V)
        assert Ps[b].tolist() == pos.tolist()
    cache.check()


def test_bf16_without_rope_stores_inputs_unchanged():
    """rope_base = 0 switches the rotation off: stored keys are the input keys, bit for bit
    (signed zeros included), and the decode output matches the oracle."""
    need_gpu()
    B, H, D, L0 = 2, 4, 128, [3, 70]
    k = W.normal_np((B, H, max(L0) + 1, D), 83)
    k[0, 0, 0, :8] = [0.0, -0.0, 0.0, -0.0, -0.0, 0.0, 1.0, -1.0]
    kd = device_tensor(k, "bf16")
    vd = device_tensor(W.normal_np((B, H, max(L0) + 1, D), 84), "bf16")
    qd = device_tensor(W.normal_np((B, H, max(L0) + 1, D), 85), "bf16")
    cache = KVCache(B, H, 128, D, dtype="bf16", rope_base=0.0)
    cache.prefill_suffix(0, None, kd[:, :, :max(L0)].contiguous(), vd[:, :, :max(L0)].contiguous(), seqlen=L0,
                         out=False)
    idx = torch.tensor(L0, device="cuda")
    sel = lambda x: x[torch.arange(B, device="cuda"), :, idx][:, :, None, :].contiguous()
    out = to_np(cache.append_attend(0, sel(qd), sel(kd), sel(vd)))
    Ks, _, _ = cache.storage(0)
    kn, vn, qn = to_np(kd), to_np(vd), to_np(qd)
    for b in range(B):
        n = L0[b] + 1
        assert torch.equal(Ks[b, :, :n].view(torch.int16).cpu(), kd[b, :, :n].view(torch.int16).cpu())
        ref = A.decode_steps_reference(qn[b, :, L0[b]][None], kn[b, :, :n], vn[b, :, :n], L0[b], 0, "bf16")
        assert np.abs(out[b, :, 0] - ref[0]).max() <= TOL["bf16"]


@pytest.mark.parametrize("Hkv,split_rows", [(8, 0), (2, 64), (1, 128)])
def test_fused_and_separate_decode_steps_agree(Hkv, split_rows):
    """One launch per step (append + attend + merge + commit) against the separate
    kernels of the same m16n8k16 decode kernel: both match the oracle; stored rows,
    positions and lengths are identical.  (With 32 query heads per key/value head the
    fused step otherwise runs on the tensor-core kernel, whose bf16 rounding points
    differ: it is compared with the oracle and this path in its own test.)"""
    L0, steps = [1, 64, 257, 100], 3
    caches, outs = [], []
    for fused in (True, False):
        cache, o, qkv = run_decode("bf16", 128, 32, Hkv, L0, steps, C=400, split_rows=split_rows, fused=fused,
                                   tc=False)
        check_against_oracle("bf16", cache, o, qkv, L0, steps)
        caches.append(cache)
        outs.append(np.stack(o))
    for x, y in zip(storage_np(caches[0]), storage_np(caches[1])):
        np.testing.assert_array_equal(x, y)
    assert caches[0].get_lengths(0) == caches[1].get_lengths(0)
    assert np.abs(outs[0] - outs[1]).max() < 5e-3


@pytest.mark.parametrize("Hq,Hkv", [(32, 32), (32, 1)])
def test_steps_fed_from_a_copy_stream_match_resident_inputs(Hq, Hkv):
    """Decode steps whose inputs arrive on another stream (pinned host -> device copies,
    double-buffered, ordered by events) give the results of steps on resident inputs:
    a decode launch must never run ahead of the event wait that precedes it."""
    need_gpu()
    B, D, steps = 64, 128, 12
    L0 = np.random.default_rng(5).integers(1, 400, size=B).tolist()
    T = max(L0) + steps
    qd, kd, vd = (device_tensor(W.normal_np((B, H, T, D), 80 + i), "bf16") for i, H in enumerate((Hq, Hkv, Hkv)))
    idx = lambda i: torch.tensor([l + i for l in L0], device="cuda")
    rows = lambda x, i: x[torch.arange(B, device="cuda"), :, idx(i)][:, :, None, :].contiguous()
    caches = []
    for _ in range(2):
        c = KVCache(B, Hq, 512, D, heads_kv=Hkv, rope_base=BASE)
        c.prefill_suffix(0, None, kd[:, :, :max(L0)].contiguous(), vd[:, :, :max(L0)].contiguous(),
                         seqlen=L0, out=False)
        caches.append(c)
    # resident inputs
    want = [caches[0].append_attend(0, rows(qd, i), rows(kd, i), rows(vd, i)) for i in range(steps)]
    # the same steps fed through a copy stream from pinned host memory, two device buffers
    host = [[rows(x, i).cpu().pin_memory() for x in (qd, kd, vd)] for i in range(steps)]
    dev = [[torch.empty_like(t, device="cuda") for t in host[0]] for _ in range(2)]
    outs = torch.empty((steps,) + tuple(want[0].shape), dtype=torch.float32, device="cuda")
    compute, copy = torch.cuda.current_stream(), torch.cuda.Stream()
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    copy.wait_stream(compute)
    for i in range(steps):
        s = i % 2
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(consumed[s])
            for d, h in zip(dev[s], host[i]):
                d.copy_(h, non_blocking=True)
            uploaded[s].record(copy)
        compute.wait_event(uploaded[s])
        caches[1].append_attend(0, *dev[s], out=outs[i], stream=compute)
        consumed[s].record(compute)
    torch.cuda.synchronize()
    for i in range(steps):
        assert torch.equal(outs[i], want[i]), i
    for x, y in zip(storage_np(caches[0]), storage_np(caches[1])):
        np.testing.assert_array_equal(x, y)
    for c in caches:
        c.check()


@pytest.mark.parametrize("Hkv", [32, 1])
def test_dependent_launch_option_changes_no_result(Hkv):
    """KVC_OPT_DECODE_PDL only changes how consecutive decode launches overlap: outputs,
    stored rows and lengths are identical with it on and off."""
    need_gpu()
    B, Hq, D, steps = 16, 32, 128, 6
    L0 = np.random.default_rng(9).integers(1, 700, size=B).tolist()
    T = max(L0) + steps
    qd, kd, vd = (device_tensor(W.normal_np((B, H, T, D), 95 + i), "bf16") for i, H in enumerate((Hq, Hkv, Hkv)))
    idx = lambda i: torch.tensor([l + i for l in L0], device="cuda")
    rows = lambda x, i: x[torch.arange(B, device="cuda"), :, idx(i)][:, :, None, :].contiguous()
    outs = []
    caches = []
    for pdl in (1, 0):
        c = KVCache(B, Hq, 1024, D, heads_kv=Hkv, rope_base=BASE)
        c.set_option(L.OPT_DECODE_PDL, pdl)
        c.prefill_suffix(0, None, kd[:, :, :max(L0)].contiguous(), vd[:, :, :max(L0)].contiguous(),
                         seqlen=L0, out=False)
        outs.append([c.append_attend(0, rows(qd, i), rows(kd, i), rows(vd, i)) for i in range(steps)])
        caches.append(c)
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    assert caches[0].get_lengths(0) == caches[1].get_lengths(0)
    for x, y in zip(storage_np(caches[0]), storage_np(caches[1])):
        np.testing.assert_array_equal(x, y)
    for c in caches:
        c.check()


@pytest.mark.gpu
def test_bound_append_attend_equals_the_plain_call():
    """KVCache.bind_append_attend (descriptors marshalled once, the bench's loop) enqueues the
    same kvc_append_attend call: outputs and stored rows equal the plain call's bit for bit,
    and the bound call keeps working when the tensors' contents change between steps."""
    need_gpu()
    B, Hq, Hkv, D, steps, C = 6, 8, 2, 128, 3, 96
    L0 = [0, 5, 17, 40, 64, 70]
    q = W.normal_np((steps, B, Hq, 1, D), 11)
    k = W.normal_np((steps, B, Hkv, 1, D), 12)
    v = W.normal_np((steps, B, Hkv, 1, D), 13)
    pre_k = W.normal_np((B, Hkv, max(L0), D), 14)
    pre_v = W.normal_np((B, Hkv, max(L0), D), 15)
    results = []
    for bound in (False, True):
        cache = KVCache(B, Hq, C, D, heads_kv=Hkv, dtype="bf16", rope_base=BASE)
        cache.prefill_suffix(0, None, device_tensor(pre_k, "bf16"), device_tensor(pre_v, "bf16"), seqlen=L0,
                             out=False)
        qi, ki, vi = (torch.empty((B, H, 1, D), dtype=torch.bfloat16, device="cuda") for H in (Hq, Hkv, Hkv))
        out = torch.empty((B, Hq, 1, D), dtype=torch.float32, device="cuda")
        call = cache.bind_append_attend(0, qi, ki, vi, out) if bound else None
        outs = []
        for i in range(steps):
            qi.copy_(device_tensor(q[i], "bf16"))
            ki.copy_(device_tensor(k[i], "bf16"))
            vi.copy_(device_tensor(v[i], "bf16"))
            if bound:
                call()
            else:
                cache.append_attend(0, qi, ki, vi, out=out)
            outs.append(to_np(out).copy())
        torch.cuda.synchronize()
        Ks, Vs, _ = storage_np(cache)
        results.append((np.stack(outs), Ks, Vs, cache.get_lengths(0)[0]))
        cache.check()
    (o0, k0, v0, l0), (o1, k1, v1, l1) = results
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(k0, k1)
    np.testing.assert_array_equal(v0, v1)
    assert l0 == l1 == [l + steps for l in L0]
