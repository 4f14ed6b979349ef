"""Parity at the full workload sizes, in the launch configuration bench.py times.

The workloads are built by bench.py's own classes (same seeds, same automatic
split plans and kernels).  The oracle recomputes sampled lanes / rows one by
one; lengths, positions and cuts are checked exhaustively, stored key and value
rows bit-exactly on the sampled lanes.  Before the timed step runs, every
storage row past a length is poisoned (keys 0, values 1e4), and every sampled
output row must also meet the relative-error guard, which -- unlike the max-abs
contract at these context lengths -- fails on a dropped key tile or a split
merged twice (tests/test_parity_power.py).
"""
import gc

import numpy as np
import pytest
import torch

import bench
from gpu_helpers import TOL, assert_close, need_gpu, to_np
from oracle import attention as A
from oracle import prefix as P

pytestmark = pytest.mark.gpu
BASE = 10000.0


def _free(*objs):
    for o in objs:
        del o
    gc.collect()
    torch.cuda.empty_cache()


def _sample_lanes(L0, n):
    order = np.argsort(L0)
    picks = [int(order[0]), int(order[-1])] + [int(b) for b in order[1:-1][:: max(1, len(order) // n)]]
    return sorted(set(picks))[:n]


@pytest.mark.parametrize("name,n_lanes", [("mha_decode", 16), ("gqa_decode", 8), ("mqa_decode", 8)])
def test_decode_workload_sampled_lanes(name, n_lanes):
    need_gpu()
    wb = bench.DecodeBench(name, torch.device("cuda", 0))
    wb.cache.poison()               # rows past the old lengths: keys 0, values 1e4
    wb.step()                       # truncate to the old lengths + every decode step, as timed
    torch.cuda.synchronize()
    c = wb.cfg
    G = c["Hq"] // c["Hkv"]
    lens, nexts = wb.cache.get_lengths(0)
    assert lens == (wb.L0 + c["steps"]).tolist() and nexts == lens
    out = wb.out.double().cpu().numpy()                       # [steps, B, H_q, 1, d]
    K, V, Ps = wb.cache.storage(0)
    worst = 0.0
    for b in _sample_lanes(wb.L0, n_lanes):
        g = (b * 7) % c["Hkv"]
        L0 = int(wb.L0[b])
        n = L0 + c["steps"]
        k = np.concatenate([to_np(wb.k_prefix[b, g, :L0]), to_np(wb.k[:, b, g, 0])])[None]
        v = np.concatenate([to_np(wb.v_prefix[b, g, :L0]), to_np(wb.v[:, b, g, 0])])[None]
        q = to_np(wb.q[:, b, g * G:(g + 1) * G, 0])
        ref = A.decode_steps_reference(q, k, v, L0, BASE, "bf16")
        worst = max(worst, assert_close(out[:, b, g * G:(g + 1) * G, 0], ref, "bf16", b))
        Ks, Vs = A.stored_rows(k, v, np.arange(n)[None], BASE, "bf16")
        np.testing.assert_array_equal(to_np(K[b, g, :n]), Ks[0])
        np.testing.assert_array_equal(to_np(V[b, g, :n]), Vs[0])
        assert Ps[b, :n].cpu().numpy().tolist() == list(range(n))
    assert worst <= TOL["bf16"], worst
    wb.cache.check()
    _free(wb)


def test_suffix_workload_sampled_rows():
    need_gpu()
    wb = bench.SuffixBench(torch.device("cuda", 0))
    # the timed step (kvc_lcp per sequence + truncate + suffix chunk) with the rows past
    # the cuts poisoned between the truncate and the chunk
    from kv_cache_append_rope_gb300 import kvc
    wb.cache.truncate([kvc.lcp(wb.cached[b], wb.query[b]) for b in range(wb.cfg["B"])])
    wb.cache.poison()
    wb.cache.prefill_suffix(0, wb.q, wb.k, wb.v, seqlen=wb.seqlen, out=wb.out)
    torch.cuda.synchronize()
    c = wb.cfg
    B, T = c["B"], wb.T
    # cuts: the library's LCP equals the oracle's on every sequence, and equals the edit position
    for b in range(B):
        assert wb.cuts[b] == P.lcp_cut(wb.cached[b].tolist(), wb.query[b].tolist()) == int(wb.edit[b])
    lens, nexts = wb.cache.get_lengths(0)
    assert lens == [T] * B and nexts == [T] * B
    K, V, Ps = wb.cache.storage(0)
    pos = Ps.cpu().numpy()
    for b in range(B):
        assert pos[b, :T].tolist() == list(range(T))
    out = wb.out
    rng = np.random.default_rng(0)
    worst = 0.0
    for b, h in [(int(np.argmin(wb.cuts)), 3), (int(np.argmax(wb.cuts)), 17)]:
        cut, S = wb.cuts[b], wb.seqlen[b]
        rows = np.unique(np.concatenate([np.arange(min(128, S)), np.arange(max(0, S - 128), S),
                                         rng.integers(0, S, 256)]))
        k = np.concatenate([to_np(wb.k_prefix[b, h, :cut]), to_np(wb.k[b, h, :S])])[None]
        v = np.concatenate([to_np(wb.v_prefix[b, h, :cut]), to_np(wb.v[b, h, :S])])[None]
        q = to_np(wb.q[b, h:h + 1, :S])
        ref = A.suffix_reference(q, k, v, np.arange(T), cut, BASE, "bf16", rows=rows)[0]
        got = out[b, h, torch.as_tensor(rows, device="cuda")].double().cpu().numpy()
        worst = max(worst, assert_close(got, ref, "bf16", (b, h)))
        Ks, Vs = A.stored_rows(k, v, np.arange(T)[None], BASE, "bf16")
        np.testing.assert_array_equal(to_np(K[b, h, :T]), Ks[0])
        np.testing.assert_array_equal(to_np(V[b, h, :T]), Vs[0])
    assert worst <= TOL["bf16"], worst
    wb.cache.check()
    _free(wb)
