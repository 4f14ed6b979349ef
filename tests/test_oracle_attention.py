"""Pins of oracle.attention: torch's SDPA (float64, CPU), closed-form special
cases, and incremental == full-prefix recomputation."""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle.rope import rotate
from oracle.storage import round_to


def test_causal_attention_matches_torch_sdpa():
    rng = np.random.default_rng(10)
    T, d = 37, 16
    Q, K, V = (rng.normal(size=(T, d)) for _ in range(3))
    mine = A.causal_attention(Q, K, V, np.arange(T))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], is_causal=True)[0]
    np.testing.assert_allclose(mine, ref.numpy(), atol=1e-13)


def test_suffix_mask_matches_torch_sdpa_with_explicit_mask():
    rng = np.random.default_rng(11)
    T, cut, d = 29, 11, 8
    Q = rng.normal(size=(T - cut, d))
    K, V = rng.normal(size=(T, d)), rng.normal(size=(T, d))
    mine = A.causal_attention(Q, K, V, cut + np.arange(T - cut))
    mask = torch.arange(T)[None, :] <= (cut + torch.arange(T - cut))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], attn_mask=mask[None])[0]
    np.testing.assert_allclose(mine, ref.numpy(), atol=1e-13)


def test_single_row_returns_its_value_and_equal_keys_average():
    rng = np.random.default_rng(12)
    v = rng.normal(size=(1, 8))
    w, o = A.attend_newest(rng.normal(size=8), rng.normal(size=(1, 8)), v)
    assert w.tolist() == [1.0]
    np.testing.assert_array_equal(o, v[0])
    K = np.tile(rng.normal(size=8), (5, 1))
    V = rng.normal(size=(5, 8))
    w, o = A.attend_newest(rng.normal(size=8), K, V)
    np.testing.assert_allclose(w, np.full(5, 0.2), atol=1e-15)
    np.testing.assert_allclose(o, V.mean(0), atol=1e-15)


def test_softmax_is_stable_for_large_scores():
    K = np.array([[1000.0, 0.0], [999.0, 0.0], [-1000.0, 0.0]])
    w, o = A.attend_newest(np.array([100.0, 0.0]), K, np.eye(3)[:, :2])
    assert np.all(np.isfinite(w)) and abs(w.sum() - 1.0) < 1e-15
    assert w[0] == pytest.approx(1.0) and w[2] == 0.0


@pytest.mark.parametrize("dtype", ["f64", "f32", "bf16"])
@pytest.mark.parametrize("heads", [(4, 4), (4, 2), (4, 1)])
def test_incremental_equals_full_prefix(dtype, heads):
    Hq, Hkv = heads
    B, C, d, L0, steps = 3, 24, 8, [0, 5, 11], 6
    rng = np.random.default_rng(13)
    cache = A.LayerCache(B, Hq, Hkv, C, d, dtype, 10000.0)
    kh = rng.normal(size=(B, Hkv, C, d))
    vh = rng.normal(size=(B, Hkv, C, d))
    qh = rng.normal(size=(B, Hq, C, d))
    S = max(L0)
    cache.prefill(qh[:, :, :S], kh[:, :, :S], vh[:, :, :S], [0] * B,
                  [min(l, S) for l in L0])
    outs = []
    for i in range(steps):
        step_k = np.stack([kh[b, :, L0[b] + i] for b in range(B)])
        step_v = np.stack([vh[b, :, L0[b] + i] for b in range(B)])
        step_q = np.stack([qh[b, :, L0[b] + i] for b in range(B)])
        outs.append(cache.append_attend(step_q, step_k, step_v))
    for b in range(B):
        n = L0[b] + steps
        ref = A.decode_steps_reference(
            np.stack([qh[b, :, L0[b] + i] for i in range(steps)]), kh[b, :, :n], vh[b, :, :n],
            L0[b], 10000.0, dtype)
        got = np.stack([o[b] for o in outs])
        np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)
        K, V = A.stored_rows(kh[b, :, :n], vh[b, :, :n], np.arange(n)[None], 10000.0, dtype)
        np.testing.assert_array_equal(cache.logical_keys(b), K)
        np.testing.assert_array_equal(cache.logical_values(b), V)
        assert cache.positions[b, :n].tolist() == list(range(n))


def test_chunk_equals_repeated_decode_and_full_prefill():
    rng = np.random.default_rng(14)
    Hq, Hkv, d, T, cut = 4, 2, 8, 20, 7
    q, k, v = rng.normal(size=(1, Hq, T, d)), rng.normal(size=(1, Hkv, T, d)), rng.normal(size=(1, Hkv, T, d))
    a = A.LayerCache(1, Hq, Hkv, T, d, "bf16", 10000.0)
    a.prefill(q[:, :, :cut], k[:, :, :cut], v[:, :, :cut], [0], [cut])
    chunk = a.prefill(q[:, :, cut:], k[:, :, cut:], v[:, :, cut:], [cut], [T - cut])
    b = A.LayerCache(1, Hq, Hkv, T, d, "bf16", 10000.0)
    b.prefill(q[:, :, :cut], k[:, :, :cut], v[:, :, :cut], [0], [cut])
    dec = np.stack([b.append_attend(q[:, :, i], k[:, :, i], v[:, :, i]) for i in range(cut, T)], axis=2)
    np.testing.assert_allclose(chunk, dec, atol=1e-12)
    ref = A.suffix_reference(q[0, :, cut:], k[0], v[0], np.arange(T), cut, 10000.0, "bf16")
    np.testing.assert_allclose(chunk[0], ref, atol=1e-12)
    # cut = 0: the chunk is a plain causal prefill
    c = A.LayerCache(1, Hq, Hkv, T, d, "f64", 10000.0)
    full = c.prefill(q, k, v, [0], [T])
    for h in range(Hq):
        g = h // 2
        qr = rotate(q[0, h], np.arange(T), 10000.0)
        kr = rotate(k[0, g], np.arange(T), 10000.0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qr)[None], torch.from_numpy(kr)[None], torch.from_numpy(v[0, g])[None],
            is_causal=True)[0].numpy()
        np.testing.assert_allclose(full[0, h], ref, atol=1e-13)


def test_gqa_reduces_to_mha_on_replicated_heads():
    rng = np.random.default_rng(15)
    Hq, d, t = 8, 16, 9
    q = rng.normal(size=(Hq, d))
    k1, v1 = rng.normal(size=(1, t, d)), rng.normal(size=(1, t, d))
    mqa = A.decode_reference(q, t - 1, k1, v1, np.arange(t), 10000.0, "f64")
    mha = A.decode_reference(q, t - 1, np.repeat(k1, Hq, 0), np.repeat(v1, Hq, 0), np.arange(t), 10000.0, "f64")
    np.testing.assert_array_equal(mqa, mha)


def test_stale_positions_change_the_suffix():
    rng = np.random.default_rng(16)
    Hq, d, T, cut = 2, 8, 12, 4
    q, k, v = rng.normal(size=(Hq, T - cut, d)), rng.normal(size=(Hq, T, d)), rng.normal(size=(Hq, T, d))
    good = A.suffix_reference(q, k, v, np.arange(T), cut, 10000.0, "f64")
    stale_pos = np.concatenate([np.arange(cut), 8 + np.arange(T - cut)])
    stale = A.suffix_reference(q, k, v, stale_pos, cut, 10000.0, "f64")
    assert np.abs(stale - good).max() > 1e-12
    # shifting every position by one constant leaves attention unchanged (relative RoPE)
    shifted = A.suffix_reference(q, k, v, np.arange(T) + 100, cut, 10000.0, "f64")
    np.testing.assert_allclose(shifted, good, atol=1e-10)


def test_layer_cache_rejects_full_without_change():
    c = A.LayerCache(1, 1, 1, 2, 2, "f64", 10000.0)
    x = np.ones((1, 1, 2))
    c.append_attend(x, x, x)
    c.append_attend(x, x, x)
    K, length = c.K.copy(), c.length.copy()
    with pytest.raises(OverflowError):
        c.append_attend(x, x, x)
    np.testing.assert_array_equal(c.K, K)
    np.testing.assert_array_equal(c.length, length)
    with pytest.raises(ValueError):
        A.LayerCache(1, 1, 1, 5, 2, max_positions=4)
