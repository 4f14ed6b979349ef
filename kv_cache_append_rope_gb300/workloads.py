"""Seeded synthetic inputs shaped like the pages' workloads.

This module draws random numbers and token ids only: it holds none of the
method's arithmetic (no rotation, no attention, no cut rule).  Both the CUDA
path (bench, GPU tests) and the oracle side (tests) take their inputs from it.

Configurations (sizes as the workloads are stated):

* fixture      1 layer, B = 1, D = 4, H = 2, d_h = 2, C = 4, f64, 3 decode calls
* prefix_reuse 2-layer single-head decoder, d = 16, vocab 32, f64, seeds 7/11/23
* mha_decode   B = 32, H = 32, d_h = 128, bf16, C = 8192, old lengths uniform in
               [1, 8191] (capped so 64 steps fit), 64 decode steps
* mha_decode_short  B = 128, H = 32, d_h = 128, bf16, C = 1024, old lengths uniform
               in [1, 256], 64 steps: short decode steps (~0.27 GB of K/V, ~40 us),
               where the gaps between launches are a visible share
* gqa_decode   B = 64, H_q = 32, H_kv = 8 or 1, d_h = 128, bf16, C = 32768,
               lengths uniform in [16384, 32767] (capped so 32 steps fit), 32 steps
* suffix       B = 8, H = 32, d_h = 128, bf16, cached prefix 16384 tokens with
               one edited id each, 512 appended ids, C = 16896
"""
import numpy as np
import torch

CONFIGS = {
    "mha_decode": dict(B=32, Hq=32, Hkv=32, D=128, C=8192, lo=1, hi=8191, steps=64, seed=3),
    "mha_decode_short": dict(B=128, Hq=32, Hkv=32, D=128, C=1024, lo=1, hi=256, steps=64, seed=3),
    "gqa_decode": dict(B=64, Hq=32, Hkv=8, D=128, C=32768, lo=16384, hi=32767, steps=32, seed=4),
    "mqa_decode": dict(B=64, Hq=32, Hkv=1, D=128, C=32768, lo=16384, hi=32767, steps=32, seed=4),
    "suffix": dict(B=8, Hq=32, Hkv=32, D=128, prefix=16384, appended=512, vocab=32000, seed=5),
}


def old_lengths(seed, B, lo, hi, capacity, steps):
    """Per-sequence old lengths, uniform over integers in [lo, min(hi, capacity - steps)]."""
    rng = np.random.default_rng(seed)
    top = min(hi, capacity - steps)
    return rng.integers(lo, top + 1, size=B).astype(np.int64)


def normal(shape, seed, dtype=torch.bfloat16, device="cuda"):
    """N(0, 1) tensor drawn by torch's generator on ``device`` from ``seed``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def normal_np(shape, seed):
    """N(0, 1) float64 array from numpy's default_rng(seed)."""
    return np.random.default_rng(seed).normal(size=shape)


def edited_histories(seed, B, prefix, appended, vocab):
    """Cached ids [B, prefix], query ids [B, prefix + appended] with one edited id.

    Cached ids are uniform in [0, vocab); the edit position e_b is uniform in
    [0, prefix - 1] and gets an id different from the cached one; the query
    continues with ``appended`` fresh uniform ids.
    """
    rng = np.random.default_rng(seed)
    cached = rng.integers(0, vocab, size=(B, prefix)).astype(np.int32)
    edit = rng.integers(0, prefix, size=B)
    query = np.concatenate([cached, rng.integers(0, vocab, size=(B, appended)).astype(np.int32)], axis=1)
    for b in range(B):
        new = int(rng.integers(0, vocab - 1))
        query[b, edit[b]] = new if new < cached[b, edit[b]] else new + 1
    return cached, query, edit


# ---- small fixed workloads -------------------------------------------------

def fixture_head_rows():
    """Per-head projected rows [3 steps, H = 2, d_h = 2] (q = k = v), unrotated.

    The chapter-37 fixture prints every rotated key, value, weight and output
    but not its weights or inputs; these rows reproduce that trace at the
    attention level: head 0 (cos p, -sin p) and head 1 (1, 0), (0, 1), (1, 1)
    for p = 0, 1, 2.
    """
    rows = np.zeros((3, 2, 2))
    for p in range(3):
        rows[p, 0] = (np.cos(p), -np.sin(p))
    rows[:, 1] = [(1.0, 0.0), (0.0, 1.0), (1.0, 1.0)]
    return rows


def fixture_random_variant(seed=0, steps=3, D=4):
    """Wq, Wk, Wv, Wo ~ N(0, 1/D) then inputs x ~ N(0, 1) [steps, D], from default_rng(seed)."""
    rng = np.random.default_rng(seed)
    std = np.sqrt(1.0 / D)
    Wq, Wk, Wv, Wo = (rng.normal(0.0, std, (D, D)) for _ in range(4))
    x = rng.normal(0.0, 1.0, (steps, D))
    return Wq, Wk, Wv, Wo, x


def toy_decoder_weights(seed, d=16, vocab=32, layers=2):
    """Embedding E [vocab, d] then (Wq, Wk, Wv, Wo) per layer, all ~ N(0, 1/16), default_rng(seed)."""
    rng = np.random.default_rng(seed)
    std = np.sqrt(1.0 / 16.0)
    E = rng.normal(0.0, std, (vocab, d))
    W = [tuple(rng.normal(0.0, std, (d, d)) for _ in range(4)) for _ in range(layers)]
    return E, W
