"""Pins of oracle.prefix and oracle.toy_decoder against the [LCP5] table,
brute force and cached == recomputed."""
import os

import numpy as np
import pytest

from golden_data import lcp5_table
from oracle import prefix as P
from oracle.toy_decoder import ToyDecoder
from kv_cache_append_rope_gb300.workloads import toy_decoder_weights

CACHED = list(range(1, 9))
TAIL = [9, 10, 11, 12]


def query_for(condition):
    """Query ids of each in-scope condition (reading of the table's row names)."""
    if condition == "append":
        return CACHED, CACHED + TAIL
    if condition == "edit_first":
        return CACHED, [20] + CACHED[1:] + TAIL
    if condition == "edit_fifth":
        return CACHED, CACHED[:4] + [20] + CACHED[5:] + TAIL
    if condition == "edit_eighth":
        return CACHED, CACHED[:7] + [20] + TAIL
    if condition == "shortened":
        return CACHED, CACHED[:4]
    if condition == "branch_append":
        branch = [1, 2, 3, 4, 5, 20, 21, 22]
        return branch, branch + TAIL
    if condition == "full_hit":
        return CACHED, list(CACHED)
    raise KeyError(condition)


def test_table_cuts_and_projection_counts():
    table, example = lcp5_table()
    assert P.lcp_cut(example["example_old"], example["example_new"]) == example["example_cut"][0]
    for cond, row in table.items():
        if not row["in_scope"]:
            continue
        cached, query = query_for(cond)
        assert len(query) == row["query_len"]
        cut = P.lcp_cut(cached, query)
        assert cut == row["cut"], cond
        assert P.projection_rows(2, len(query), cut) == row["rows"]
        assert P.projection_rows(2, len(query), 0) == row["full_rows"]
    # full-cache hit: cut stops one short of the query so the last token is recomputed
    assert P.lcp_cut(*query_for("full_hit")) == 7
    assert P.projection_rows(2, 8, 7) == 6


def test_lcp_brute_force_against_commonprefix():
    rng = np.random.default_rng(20)
    for _ in range(3000):
        a = rng.integers(0, 3, rng.integers(0, 9)).tolist()
        b = rng.integers(0, 3, rng.integers(1, 9)).tolist()
        n = len(os.path.commonprefix([a, b]))
        assert P.longest_common_prefix(a, b) == n
        assert P.lcp_cut(a, b) == min(n, len(b) - 1)


def test_lcp_edge_cases():
    assert P.lcp_cut([], [5, 6]) == 0
    assert P.lcp_cut([1, 2, 3], [1, 9, 3]) == 1          # equal again after a difference: not counted
    with pytest.raises(ValueError):
        P.lcp_cut([1, 2], [])
    with pytest.raises(TypeError):
        P.lcp_cut([1, 2], [1.0, 2])
    with pytest.raises(TypeError):
        P.lcp_cut([1, 2], [True, 2])


def test_truncate_keeps_prefix_and_sets_next_position():
    k = np.arange(24, dtype=float).reshape(6, 4)
    cache = {"next_position": 6, "layers": [(k, k + 1, np.arange(6))] * 2}
    t = P.truncate(cache, 4)
    assert t["next_position"] == 4
    for kk, vv, pp in t["layers"]:
        np.testing.assert_array_equal(kk, k[:4])
        np.testing.assert_array_equal(vv, k[:4] + 1)
        assert pp.tolist() == [0, 1, 2, 3]
        assert kk.base is None                             # a copy, not a view
    with pytest.raises(ValueError):
        P.truncate(cache, 7)


CONDITIONS = ["append", "edit_first", "edit_fifth", "edit_eighth", "shortened", "branch_append", "full_hit"]


@pytest.mark.parametrize("seed", [7, 11, 23])
@pytest.mark.parametrize("condition", CONDITIONS)
def test_toy_decoder_reuse_equals_recompute_and_stale_control(seed, condition):
    model = ToyDecoder(*toy_decoder_weights(seed))
    cached, query = query_for(condition)
    _, cache = model.forward_full(cached)
    cut = P.lcp_cut(cached, query)
    full_h, full_cache = model.forward_full(query)
    reused = P.truncate(cache, cut)
    h, new_cache = model.chunk(query[cut:], reused)
    err = np.abs(h - full_h[cut:]).max()
    assert err <= 1e-12
    for (k, v, p), (fk, fv, fp) in zip(new_cache["layers"], full_cache["layers"]):
        assert np.abs(k - fk).max() <= 1e-12 and np.abs(v - fv).max() <= 1e-12
        assert p.tolist() == fp.tolist() == list(range(len(query)))
    # negative control: same truncation, next_position left at the old length
    stale = P.truncate(cache, cut)
    stale["next_position"] = len(cached)
    hs, _ = model.chunk(query[cut:], stale)
    stale_err = np.abs(hs - full_h[cut:]).max()
    if cut == len(cached):
        assert stale_err == 0.0                           # plain append: nothing is stale
    else:
        assert stale_err > 1e-12


def test_toy_decoder_is_causal():
    model = ToyDecoder(*toy_decoder_weights(7))
    a, _ = model.forward_full([1, 2, 3, 4, 5, 6])
    b, _ = model.forward_full([1, 2, 3, 30, 31, 0])
    np.testing.assert_array_equal(a[:3], b[:3])
    assert np.abs(a[3:] - b[3:]).min() > 0
