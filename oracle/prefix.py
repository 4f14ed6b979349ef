"""Longest-common-prefix reuse: cut, truncation, projection counts.

[LCP5] (huhohoo.com/docs/llm/longest-prefix-reuse):

* section "先看一次历史编辑": only the contiguous run of equal ids starting at
  the first token is reusable; ids that agree again after a difference do not
  count.
* section "查询流程与缓存所有权": token ids must be non-empty integers (a float
  1.0 must not match the integer 1); the query is cut at
  cut <= len(query) - 1 so that at least the last token is recomputed.
* listing under "哪些东西必须一起裁剪": every layer keeps k[:cut], v[:cut],
  positions[:cut] and next_position becomes cut.
* table and text under "27 例得到的计算量与误差": projection rows of the
  continuation are layers x 3 (Q, K, V) x (len(query) - cut).
* section "为什么滑窗部分命中必须回退": the conservative reuse rule of a
  sliding-window cache (lcp_cut_window).
"""

import numbers

import numpy as np


def _validate_ids(ids, what):
    if len(ids) == 0:
        raise ValueError(f"{what} token ids must be non-empty")
    for t in ids:
        if isinstance(t, (bool, np.bool_)) or not isinstance(t, (numbers.Integral, np.integer)):
            raise TypeError(f"{what} token ids must be integers, got {t!r}")


def longest_common_prefix(cached_ids, query_ids):
    """Length of the run of equal ids from index 0."""
    n = 0
    for a, b in zip(cached_ids, query_ids):
        if a != b:
            break
        n += 1
    return n


def lcp_cut(cached_ids, query_ids):
    """cut = min(LCP(cached, query), len(query) - 1).

    An empty cached sequence gives cut 0; an empty query or a non-integer id
    is an error.
    """
    _validate_ids(query_ids, "query")
    if len(cached_ids):
        _validate_ids(cached_ids, "cached")
    return min(longest_common_prefix(cached_ids, query_ids), len(query_ids) - 1)


def lcp_cut_window(cached_ids, query_ids, window):
    """The cut for a sliding-window cache ([LCP5] "为什么滑窗部分命中必须回退").

    A window cache no longer holds the early rows of its history, so a prefix
    of it cannot stand for a prefix of the history: the window is reused only
    when the whole cached sequence matches and the query continues past it
    (cut = len(cached)); any partial hit recomputes from the start (cut = 0).
    ``window`` == 0 is the full-attention rule (lcp_cut).
    """
    if not window:
        return lcp_cut(cached_ids, query_ids)
    _validate_ids(query_ids, "query")
    if len(cached_ids):
        _validate_ids(cached_ids, "cached")
    n = len(cached_ids)
    if longest_common_prefix(cached_ids, query_ids) == n and len(query_ids) > n:
        return n
    return 0


def projection_rows(layers, query_len, cut):
    """Rows projected by the continuation: layers x 3 x (query_len - cut)."""
    return layers * 3 * (query_len - cut)


def truncate(cache, cut):
    """Truncated copy of a cache dict {'next_position', 'layers': [(k, v, positions)]}.

    k/v are [..., T, d] arrays (rows on the second-to-last axis), positions [T].
    """
    layers = []
    for k, v, pos in cache["layers"]:
        if cut > pos.shape[-1]:
            raise ValueError("cut exceeds the cached length")
        layers.append((k[..., :cut, :].copy(), v[..., :cut, :].copy(), pos[..., :cut].copy()))
    return {"next_position": cut, "layers": layers}
