"""Newest-query and causal attention over a RoPE key/value cache, float64.

Definitions followed (cited by page title and section / listing title):

* [Ch37] listing "Evaluate one newest query across the retained rows plus the
  candidate key/value row before committing the append": score s_j =
  q . k_j / sqrt(d_h) for every retained row and the candidate row; weights are
  a numerically stable softmax (max subtracted, [Ch37] "Bind the state,
  calculate completely, then commit"); the output is sum_j a_j v_j.
* [Ch37] "Append along the position axis": K_{1:t} = [K_{1:t-1}; k_t],
  V_{1:t} = [V_{1:t-1}; v_t]; the key is rotated at the zero-based old length,
  the value is not rotated, the query is not stored.
* [Ch37] "From causal attention to managed LLM inference state": the
  reference is the full-prefix masked scaled dot-product attention of
  "Attention Is All You Need".
* [LCP5] section "先看一次历史编辑" and the listing under
  "哪些东西必须一起裁剪": after truncation to ``cut`` the suffix is computed
  against the retained prefix, continuing at position ``cut``.

Readings where the pages are silent:

* The cache holds rows in its storage dtype, so attention reads the rounded
  rotated key and rounded value; the query is rotated in float64 and not
  rounded (it is never stored).
* Grouped / multi-query attention (the pages cite Shazeer's multi-query
  attention only): query head h reads key/value head h // G, G = H_q / H_kv.
* The causal mask of a suffix chunk is by slot index: suffix row i (slot
  cut + i) sees slots 0 .. cut + i, whatever positions were recorded.
* Sliding window ([LCP5] "为什么滑窗部分命中必须回退": a window-4 cache keeps
  only the last four rows, positions 4..7 of 8): with window W >= 1 the row
  at slot s sees only slots s - W + 1 .. s (its W most recent rows, itself
  included); W = 0 means no window.
"""

import math

import numpy as np

from .rope import rotate
from .storage import round_to


def stable_softmax(scores):
    """Softmax over the last axis with the maximum subtracted first."""
    s = np.asarray(scores, dtype=np.float64)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attend_newest(q, K, V):
    """One query row ``q`` [d] against key/value rows ``K``, ``V`` [t, d].

    Returns (weights [t], output [d]).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        raise ValueError("attention needs at least one key row")
    scale = 1.0 / math.sqrt(q.shape[-1])
    w = stable_softmax((K @ q) * scale)
    return w, w @ V


def causal_attention(Q, K, V, query_slots, window=0):
    """Masked scaled dot-product attention.

    ``Q`` [n, d] query rows, ``K``/``V`` [T, d] key/value rows in slot order;
    query row i attends slots 0 .. query_slots[i] (inclusive), and with
    ``window`` W >= 1 only slots query_slots[i] - W + 1 and later.  Returns [n, d].
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    slots = np.asarray(query_slots, dtype=np.int64)
    scale = 1.0 / math.sqrt(Q.shape[-1])
    s = (Q @ K.T) * scale
    j = np.arange(K.shape[0])[None, :]
    visible = j <= slots[:, None]
    if window:
        visible &= j > slots[:, None] - window
    s = np.where(visible, s, -np.inf)
    return stable_softmax(s) @ V


def kv_head_of(h, heads_q, heads_kv):
    """Key/value head read by query head ``h`` (contiguous groups)."""
    if heads_q % heads_kv:
        raise ValueError("query heads must be a multiple of key/value heads")
    return h // (heads_q // heads_kv)


def stored_rows(k_unrot, v_unrot, positions, base, dtype):
    """Cache contents written by the append: round(rotate(k, p)), round(v).

    ``k_unrot``/``v_unrot`` [..., t, d] float64, ``positions`` broadcastable to
    [..., t].  Returns (K, V) as float64 arrays holding storage-dtype values.
    """
    K = round_to(rotate(k_unrot, positions, base), dtype)
    V = round_to(np.asarray(v_unrot, dtype=np.float64), dtype)
    return K, V


def decode_reference(q_unrot, q_position, k_unrot, v_unrot, k_positions, base, dtype):
    """One decode step recomputed from the full prefix of one sequence.

    q_unrot [H_q, d] (the new query, unrotated), q_position its position;
    k_unrot, v_unrot [H_kv, t, d] every retained row plus the new row, with
    positions k_positions [t].  Returns out [H_q, d].
    """
    q_unrot = np.asarray(q_unrot, dtype=np.float64)
    Hq = q_unrot.shape[0]
    Hkv = np.asarray(k_unrot).shape[0]
    K, V = stored_rows(k_unrot, v_unrot, np.asarray(k_positions)[None, :], base, dtype)
    qr = rotate(q_unrot, np.full(Hq, q_position), base)
    out = np.empty_like(qr)
    for h in range(Hq):
        g = kv_head_of(h, Hq, Hkv)
        out[h] = attend_newest(qr[h], K[g], V[g])[1]
    return out


def decode_steps_reference(q_steps, k_unrot, v_unrot, prefix_len, base, dtype, window=0):
    """Consecutive decode steps of one sequence, each recomputed from its prefix.

    q_steps [steps, H_q, d]: the query of step i sits at position prefix_len + i.
    k_unrot, v_unrot [H_kv, prefix_len + steps, d]: row j sits at position j.
    Step i attends rows 0 .. prefix_len + i (with ``window`` W >= 1 only the
    last W of them).  Returns [steps, H_q, d].
    """
    q_steps = np.asarray(q_steps, dtype=np.float64)
    steps, Hq, _ = q_steps.shape
    Hkv, T, _ = np.asarray(k_unrot).shape
    if T != prefix_len + steps:
        raise ValueError("key history must hold prefix_len + steps rows")
    K, V = stored_rows(k_unrot, v_unrot, np.arange(T)[None, :], base, dtype)
    out = np.empty_like(q_steps)
    for i in range(steps):
        t = prefix_len + i + 1
        lo = max(0, t - window) if window else 0
        qr = rotate(q_steps[i], np.full(Hq, t - 1), base)
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            out[i, h] = attend_newest(qr[h], K[g, lo:t], V[g, lo:t])[1]
    return out


def suffix_reference(q_unrot, k_unrot, v_unrot, positions, cut, base, dtype, rows=None, window=0):
    """Suffix-chunk attention of one sequence, by full masked recomputation.

    Slots 0 .. cut-1 are the retained prefix, slots cut .. T-1 the suffix.
    q_unrot [H_q, S, d] suffix queries (S = T - cut), k_unrot / v_unrot
    [H_kv, T, d] every row, ``positions`` [T] the position recorded for each
    slot (normally the slot index; a stale next_position shifts the suffix).
    Suffix row i is rotated at positions[cut + i] and attends slots 0 .. cut+i.
    ``rows`` optionally selects suffix rows; ``window`` as in causal_attention.
    Returns [H_q, len(rows), d].
    """
    q_unrot = np.asarray(q_unrot, dtype=np.float64)
    Hq, S, _ = q_unrot.shape
    Hkv, T, _ = np.asarray(k_unrot).shape
    positions = np.asarray(positions, dtype=np.int64)
    if S != T - cut:
        raise ValueError("suffix length must be T - cut")
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    K, V = stored_rows(k_unrot, v_unrot, positions[None, :], base, dtype)
    qr = rotate(q_unrot[:, rows], positions[cut + rows][None, :], base)
    out = np.empty((Hq, rows.size, q_unrot.shape[-1]))
    for h in range(Hq):
        g = kv_head_of(h, Hq, Hkv)
        out[h] = causal_attention(qr[h], K[g], V[g], cut + rows, window)
    return out


class LayerCache:
    """The incremental algorithm: fixed-capacity per-layer cache, float64.

    Mirrors [Ch37] listing "Own a fixed layer-bound cache, append one checked
    row, and reset logical length" for the state (buffers [B, H_kv, C, d_h]
    zero-filled, per-sequence logical length, reset to 0 without touching the
    storage) and the candidate-row scoring of the newest-query listing; adds
    per-slot positions and next_position from [LCP5].  Used to pin that the
    incremental computation equals the full-prefix recomputation.
    """

    def __init__(self, batch, heads_q, heads_kv, capacity, head_dim, dtype="f64",
                 rope_base=10000.0, max_positions=None):
        if batch <= 0:
            raise ValueError("KV cache batch size must be nonzero")
        if capacity <= 0:
            raise ValueError("KV cache capacity must be nonzero")
        self.max_positions = capacity if max_positions is None else max_positions
        if capacity > self.max_positions:
            raise ValueError("KV cache capacity exceeds RoPE position capacity")
        if heads_q % heads_kv:
            raise ValueError("query heads must be a multiple of key/value heads")
        self.B, self.Hq, self.Hkv, self.C, self.d = batch, heads_q, heads_kv, capacity, head_dim
        self.dtype, self.base = dtype, rope_base
        self.K = np.zeros((batch, heads_kv, capacity, head_dim))
        self.V = np.zeros((batch, heads_kv, capacity, head_dim))
        self.positions = np.zeros((batch, capacity), dtype=np.int64)
        self.length = np.zeros(batch, dtype=np.int64)
        self.next_position = np.zeros(batch, dtype=np.int64)

    def append_attend(self, q, k, v):
        """One decode step for every sequence: q [B, H_q, d], k/v [B, H_kv, d].

        Rotates at next_position (= old length on every path but the stale
        control), scores the stored rows plus the candidate row, then commits
        the candidate.  Raises before any state change when a sequence is full.
        """
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        if np.any(self.length >= self.C):
            raise OverflowError(f"KV cache is full at capacity {self.C}")
        out = np.empty_like(q)
        cand_k = np.empty_like(k)
        cand_v = np.empty_like(v)
        for b in range(self.B):
            p = int(self.next_position[b])
            n = int(self.length[b])
            qr = rotate(q[b], np.full(self.Hq, p), self.base)
            ck, cv = stored_rows(k[b][:, None, :], v[b][:, None, :],
                                 np.full((self.Hkv, 1), p), self.base, self.dtype)
            cand_k[b], cand_v[b] = ck[:, 0], cv[:, 0]
            for h in range(self.Hq):
                g = kv_head_of(h, self.Hq, self.Hkv)
                K = np.concatenate([self.K[b, g, :n], cand_k[b, g][None]], axis=0)
                V = np.concatenate([self.V[b, g, :n], cand_v[b, g][None]], axis=0)
                out[b, h] = attend_newest(qr[h], K, V)[1]
        for b in range(self.B):
            n = int(self.length[b])
            self.K[b, :, n] = cand_k[b]
            self.V[b, :, n] = cand_v[b]
            self.positions[b, n] = self.next_position[b]
            self.length[b] += 1
            self.next_position[b] += 1
        return out

    def prefill(self, q, k, v, start_pos, seqlen):
        """Append ``seqlen[b]`` rows per sequence and attend them causally.

        q [B, H_q, S, d], k/v [B, H_kv, S, d] (rows beyond seqlen[b] ignored);
        row i of sequence b goes to slot length[b] + i with position
        start_pos[b] + i.  Returns out [B, H_q, S, d] (zero beyond seqlen).
        """
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        seqlen = np.asarray(seqlen, dtype=np.int64)
        start_pos = np.asarray(start_pos, dtype=np.int64)
        if np.any(self.length + seqlen > self.C):
            raise OverflowError(f"KV cache is full at capacity {self.C}")
        out = np.zeros_like(q)
        for b in range(self.B):
            n, S = int(self.length[b]), int(seqlen[b])
            if S == 0:
                continue
            pos = start_pos[b] + np.arange(S)
            Kn, Vn = stored_rows(k[b, :, :S], v[b, :, :S], pos[None, :], self.base, self.dtype)
            self.K[b, :, n:n + S] = Kn
            self.V[b, :, n:n + S] = Vn
            self.positions[b, n:n + S] = pos
            qr = rotate(q[b, :, :S], pos[None, :], self.base)
            for h in range(self.Hq):
                g = kv_head_of(h, self.Hq, self.Hkv)
                out[b, h, :S] = causal_attention(qr[h], self.K[b, g, :n + S], self.V[b, g, :n + S],
                                                 n + np.arange(S))
            self.length[b] = n + S
            self.next_position[b] = start_pos[b] + S
        return out

    def truncate(self, cut):
        """[LCP5] "哪些东西必须一起裁剪": keep rows < cut, next_position = cut."""
        cut = np.asarray(cut, dtype=np.int64)
        if np.any(cut < 0) or np.any(cut > self.length):
            raise ValueError("cut must lie in [0, length]")
        self.length = cut.copy()
        self.next_position = cut.copy()

    def reset(self):
        """[Ch37] "Reset or reject without corrupting retained state"."""
        self.length[:] = 0
        self.next_position[:] = 0

    def logical_keys(self, b):
        return self.K[b, :, :self.length[b]]

    def logical_values(self, b):
        return self.V[b, :, :self.length[b]]
