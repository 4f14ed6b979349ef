"""Pins of the oracle's RoPE toy decoder (the [LCP5] model with rotary positions).

The rotary variant is checked against quantities computed another way:

* attention scores of rotated rows equal the relative-phase form
  Re(sum_j z_q,j conj(z_k,j) exp(i (p_q - p_k) theta_j)), with each interleaved
  pair (x, y) read as the complex number x + i y -- the whole decoder is rebuilt
  from that form, in complex arithmetic, and must agree to 1e-12;
* with no absolute positions left, starting the same ids at another position
  leaves every hidden state unchanged (only differences of positions enter);
* continuing from a cache equals the uncached forward of the whole sequence
  ([LCP5] section "先看一次历史编辑": retained rows do not depend on later tokens).
A dropped rotation, a wrong sign of the angle, a rotated value or a leftover
sinusoid fails one of them.
"""
import math

import numpy as np
import pytest

from kv_cache_append_rope_gb300 import workloads as W
from oracle.toy_decoder import ToyDecoder

BASE = 10000.0


def relative_phase_forward(E, Wl, ids, start, base):
    """The rotary decoder written with complex relative phases instead of rotations."""
    d = E.shape[1]
    theta = np.array([base ** (-2.0 * j / d) for j in range(d // 2)])
    pos = start + np.arange(len(ids))
    h = E[np.asarray(ids)]
    for Wq, Wk, Wv, Wo in Wl:
        q, k, v = h @ Wq, h @ Wk, h @ Wv
        zq = q[:, 0::2] + 1j * q[:, 1::2]
        zk = k[:, 0::2] + 1j * k[:, 1::2]
        phase = np.exp(1j * (pos[:, None, None] - pos[None, :, None]) * theta[None, None, :])
        s = np.real((zq[:, None, :] * np.conj(zk)[None, :, :] * phase).sum(axis=2)) / math.sqrt(d)
        s = np.where(np.tril(np.ones((len(ids), len(ids)), dtype=bool)), s, -np.inf)
        a = np.exp(s - s.max(axis=1, keepdims=True))
        a /= a.sum(axis=1, keepdims=True)
        h = h + np.tanh((a @ v) @ Wo)
    return h


@pytest.mark.parametrize("seed", [7, 11, 23])
def test_rotary_decoder_matches_relative_phase_form(seed):
    E, Wl = W.toy_decoder_weights(seed)
    ids = np.random.default_rng(seed).integers(0, 32, size=11).tolist()
    h, _ = ToyDecoder(E, Wl, rope_base=BASE).forward_full(ids)
    ref = relative_phase_forward(E, Wl, ids, 0, BASE)
    assert np.abs(h - ref).max() < 1e-12


def test_rotary_decoder_depends_only_on_position_differences():
    E, Wl = W.toy_decoder_weights(7)
    ids = [3, 1, 4, 1, 5, 9, 2, 6]
    model = ToyDecoder(E, Wl, rope_base=BASE)
    h0, _ = model.forward_full(ids)
    empty = {"next_position": 1000, "layers": [(np.zeros((0, 16)), np.zeros((0, 16)),
                                                np.zeros(0, dtype=np.int64))] * 2}
    h1, _ = model.chunk(ids, empty)
    assert np.abs(h0 - h1).max() < 1e-12
    # the sinusoidal model does depend on absolute positions (the control)
    s0, _ = ToyDecoder(E, Wl).forward_full(ids)
    s1, _ = ToyDecoder(E, Wl).chunk(ids, empty)
    assert np.abs(s0 - s1).max() > 1e-3


@pytest.mark.parametrize("cut", [1, 5, 10])
def test_rotary_decoder_continuation_equals_full_forward(cut):
    E, Wl = W.toy_decoder_weights(11)
    ids = np.random.default_rng(3).integers(0, 32, size=12).tolist()
    model = ToyDecoder(E, Wl, rope_base=BASE)
    full, _ = model.forward_full(ids)
    _, cache = model.forward_full(ids[:cut])
    rest, cache = model.chunk(ids[cut:], cache)
    assert np.abs(rest - full[cut:]).max() < 1e-12
    assert cache["next_position"] == len(ids)
    assert model.logits(full).shape == (len(ids), 32)
