"""The 2-layer single-head decoder of [LCP5], float64.

[LCP5] section "27 例得到的计算量与误差" fixes: two layers, one head, width
16, vocabulary 32, float64, sinusoidal absolute positions, tanh residual, no
training, no FFN, no LayerNorm.  The architecture itself belongs to an earlier
article of that series and is not printed, so this module takes the plainest
reading; the page publishes no weights either, so this architecture is parity
unpinned (only its internal invariants are checked):

* h = E[id] + PE(position), PE the sinusoid of "Attention Is All You Need":
  PE[p, 2i] = sin(p / 10000**(2i/d)), PE[p, 2i+1] = cos(p / 10000**(2i/d));
* per layer: q, k, v = h Wq, h Wk, h Wv (16 x 16), a = causal softmax(q k^T
  / sqrt(16)) v, h <- h + tanh(a Wo);
* the output is the final hidden state of every computed row;
* no RoPE.  The weights (E [vocab, d] and per layer Wq, Wk, Wv, Wo) are
  inputs: the tests draw them ~ N(0, 1/16) from the seeded generator module.

The RoPE variant (``rope_base`` given) is the same model with the absolute
sinusoid replaced by rotary positions, as [Ch37] "Append along the position
axis" uses them: h = E[id]; q and k of a row are rotated at the row's position
before attention, and the cache keeps the rotated keys.  Its greedy next token
reads the final hidden row through the tied vocabulary head (logits = h E^T).
With ``window`` W >= 1 every row attends only its W most recent rows ([LCP5]
"为什么滑窗部分命中必须回退" uses a window of 4).

The cache is the dict of the truncation listing under "哪些东西必须一起裁剪":
{'next_position': int, 'layers': [(k [T, d], v [T, d], positions [T])]}.
"""

import numpy as np

from .attention import causal_attention
from .rope import rotate


def sinusoidal_positions(positions, d):
    """Additive sinusoidal position rows [len(positions), d]."""
    pos = np.asarray(positions, dtype=np.float64)[:, None]
    i = np.arange(0, d, 2, dtype=np.float64)[None, :]
    ang = pos / np.power(10000.0, i / d)
    pe = np.zeros((pos.shape[0], d))
    pe[:, 0::2] = np.sin(ang)
    pe[:, 1::2] = np.cos(ang)
    return pe


class ToyDecoder:
    def __init__(self, E, W, rope_base=None, window=0):
        self.E = np.asarray(E, dtype=np.float64)
        self.W = [tuple(np.asarray(w, dtype=np.float64) for w in layer) for layer in W]
        self.vocab, self.d = self.E.shape
        self.n_layers = len(self.W)
        self.rope_base = rope_base
        self.window = window           # sliding window of W slots per row (0: none)

    def embed(self, ids, positions):
        rows = self.E[np.asarray(ids, dtype=np.int64)]
        if self.rope_base is not None:
            return rows
        return rows + sinusoidal_positions(positions, self.d)

    def logits(self, h):
        """Tied vocabulary head: scores of every id for hidden rows ``h``."""
        return np.asarray(h, dtype=np.float64) @ self.E.T

    def project(self, layer, h):
        Wq, Wk, Wv, _ = self.W[layer]
        return h @ Wq, h @ Wk, h @ Wv

    def mix(self, layer, h, attn):
        return h + np.tanh(attn @ self.W[layer][3])

    def forward_full(self, ids):
        """Uncached forward of every row; returns (hidden [n, d], cache dict)."""
        return self.chunk(ids, {"next_position": 0,
                                "layers": [(np.zeros((0, self.d)), np.zeros((0, self.d)),
                                            np.zeros(0, dtype=np.int64))] * self.n_layers})

    def chunk(self, ids, cache):
        """Continue from ``cache``: rows at positions next_position, ... .

        Returns (hidden states of the new rows [n, d], the extended cache).
        Slots of the new rows follow the retained rows; row i attends the
        retained slots and new rows 0..i.
        """
        n = len(ids)
        start = int(cache["next_position"])
        positions = start + np.arange(n)
        h = self.embed(ids, positions)
        new_layers = []
        for layer, (kc, vc, pc) in enumerate(cache["layers"]):
            q, k, v = self.project(layer, h)
            if self.rope_base is not None:
                q = rotate(q, positions, self.rope_base)
                k = rotate(k, positions, self.rope_base)
            K = np.concatenate([kc, k], axis=0)
            V = np.concatenate([vc, v], axis=0)
            a = causal_attention(q, K, V, kc.shape[0] + np.arange(n), self.window)
            h = self.mix(layer, h, a)
            new_layers.append((K, V, np.concatenate([pc, positions])))
        return h, {"next_position": start + n, "layers": new_layers}
