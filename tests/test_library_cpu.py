"""The C ABI without a GPU: library loads, exports every declared entry point,
and the host-side checks that run before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import prefix as P

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kvc.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(kvc_lib):
    names = declared_functions()
    assert len(names) >= 16
    for n in names:
        assert hasattr(kvc_lib.lib, n), n
    assert set(names) == set(kvc_lib.EXPORTS)
    assert kvc_lib.lib.kvc_abi_version() == 5


def test_debug_build_loads_and_exports_the_same_symbols(kvc_lib):
    """libkvc_debug.so (every kernel's bounds checks compiled in) has the same ABI."""
    from kv_cache_append_rope_gb300 import build
    dbg = ctypes.CDLL(build.DEBUG_LIB)
    for n in declared_functions():
        assert hasattr(dbg, n), n
    dbg.kvc_abi_version.restype = ctypes.c_int32
    assert dbg.kvc_abi_version() == 5


def test_length_query_and_no_handle_options_need_no_device(kvc_lib):
    L = kvc_lib
    ln = (ctypes.c_int32 * 1)()
    assert L.STATUS[L.lib.kvc_get_len(None, 0, ln)] == "KVC_ERR_NULL"
    assert L.STATUS[L.lib.kvc_read_rows(None, 0, None, None, None, None)] == "KVC_ERR_NULL"
    # a NULL handle accepts only the no-alloc stall arm (a host flag), every other option is refused
    assert L.STATUS[L.lib.kvc_set_option(None, L.OPT_TEST_POISON, 1)] == "KVC_ERR_NULL"


def test_status_strings(kvc_lib):
    for code, name in kvc_lib.STATUS.items():
        s = kvc_lib.status_string(code)
        assert s and s != "unknown status", name


def _create(kvc_lib, **kw):
    cfg = kvc_lib.kvc_config()
    base = dict(batch=1, heads_q=2, heads_kv=2, capacity=4, head_dim=2, layers=1, dtype=2,
                rope_max_positions=0, rope_base=10000.0, checked=0, device=0)
    base.update(kw)
    for k, v in base.items():
        setattr(cfg, k, v)
    h = ctypes.c_void_p(123)
    st = kvc_lib.lib.kvc_create_ex(ctypes.byref(cfg), ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("kw,code", [
    (dict(batch=0), "KVC_ERR_ZERO_BATCH"),
    (dict(capacity=0), "KVC_ERR_ZERO_CAPACITY"),
    (dict(capacity=5, rope_max_positions=4), "KVC_ERR_CAPACITY_EXCEEDS_POSITIONS"),
    (dict(heads_q=3, heads_kv=2), "KVC_ERR_CONFIG"),
    (dict(head_dim=3), "KVC_ERR_CONFIG"),
    (dict(dtype=7), "KVC_ERR_CONFIG"),
    (dict(window=-1), "KVC_ERR_CONFIG"),
    (dict(block_rows=32), "KVC_ERR_CONFIG"),
    (dict(block_rows=192), "KVC_ERR_CONFIG"),
    (dict(block_rows=64, blocks=-1), "KVC_ERR_CONFIG"),
    (dict(batch=2**30, heads_kv=2**30, heads_q=2**30, capacity=2**30, head_dim=256, layers=2**30), None),
])
def test_create_rejections_before_any_cuda_call(kvc_lib, kw, code):
    st, h = _create(kvc_lib, **kw)
    if code is None:
        assert kvc_lib.STATUS[st] == "KVC_ERR_ELEMENT_OVERFLOW"
    else:
        assert kvc_lib.STATUS[st] == code
    assert h.value is None                      # *out cleared, nothing allocated
    assert kvc_lib.last_error()                  # a message explains it


def test_null_arguments(kvc_lib):
    h = ctypes.c_void_p()
    assert kvc_lib.STATUS[kvc_lib.lib.kvc_create_ex(None, ctypes.byref(h))] == "KVC_ERR_NULL"
    assert kvc_lib.STATUS[kvc_lib.lib.kvc_append_attend(None, 0, None, None, None, None, None)] == "KVC_ERR_NULL"
    assert kvc_lib.STATUS[kvc_lib.lib.kvc_truncate(None, None, None)] == "KVC_ERR_NULL"
    assert kvc_lib.STATUS[kvc_lib.lib.kvc_prepare_attend(None, 0, None, None, None, None, None, None)] == "KVC_ERR_NULL"
    assert kvc_lib.STATUS[kvc_lib.lib.kvc_commit(None, None, 0, None)] == "KVC_ERR_NULL"
    assert kvc_lib.STATUS[kvc_lib.lib.kvc_sync_lengths(None)] == "KVC_ERR_NULL"
    assert kvc_lib.STATUS[kvc_lib.lib.kvc_prefill_suffix_host(None, 0, None, None, None, None, None, None, 0,
                                                             None)] == "KVC_ERR_NULL"
    kvc_lib.lib.kvc_destroy(None)


def _lcp(kvc_lib, a, b):
    cut = ctypes.c_int32(-1)
    st = kvc_lib.lib.kvc_lcp(kvc_lib.int_array(a) if a else None, len(a),
                             kvc_lib.int_array(b) if b else None, len(b), ctypes.byref(cut))
    return kvc_lib.STATUS[st], cut.value


def test_lcp_window_matches_oracle(kvc_lib):
    """kvc_lcp_window against oracle.prefix.lcp_cut_window on random small id lists."""
    rng = np.random.default_rng(21)
    for _ in range(2000):
        a = rng.integers(0, 3, rng.integers(0, 9)).tolist()
        b = rng.integers(0, 3, rng.integers(1, 9)).tolist()
        w = int(rng.integers(0, 4))
        cut = ctypes.c_int32(-1)
        st = kvc_lib.lib.kvc_lcp_window(kvc_lib.int_array(a) if a else None, len(a), kvc_lib.int_array(b), len(b),
                                        w, ctypes.byref(cut))
        assert kvc_lib.STATUS[st] == "KVC_OK"
        assert cut.value == P.lcp_cut_window(a, b, w)
    cut = ctypes.c_int32(-1)
    assert kvc_lib.STATUS[kvc_lib.lib.kvc_lcp_window(None, 0, kvc_lib.int_array([1]), 1, -1,
                                                     ctypes.byref(cut))] == "KVC_ERR_CONFIG"


def test_lcp_matches_oracle_and_table(kvc_lib):
    rng = np.random.default_rng(30)
    for _ in range(2000):
        a = rng.integers(0, 3, rng.integers(0, 10)).tolist()
        b = rng.integers(0, 3, rng.integers(1, 10)).tolist()
        st, cut = _lcp(kvc_lib, a, b)
        assert st == "KVC_OK" and cut == P.lcp_cut(a, b)
    assert _lcp(kvc_lib, list(range(1, 9)), [1, 2, 3, 4, 20, 6, 7, 8, 9, 10, 11, 12]) == ("KVC_OK", 4)
    assert _lcp(kvc_lib, list(range(1, 9)), list(range(1, 9))) == ("KVC_OK", 7)
    assert _lcp(kvc_lib, list(range(1, 9)), [1, 2, 3, 4]) == ("KVC_OK", 3)
    assert _lcp(kvc_lib, [], [5]) == ("KVC_OK", 0)
    assert _lcp(kvc_lib, [1, 2], [])[0] == "KVC_ERR_EMPTY_QUERY"


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib

    import kv_cache_append_rope_gb300._lib as L
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        L._load()
    importlib.reload(L)


def test_host_buffer_descriptors():
    """The binding of kvc_prefill_suffix_host describes CPU tensors as they are (pointer,
    dtype, rank, shape) and refuses what the call cannot take."""
    import torch

    from kv_cache_append_rope_gb300 import _lib as L
    from kv_cache_append_rope_gb300.kvc import host_tensor_desc
    t = torch.zeros((2, 4, 5, 128), dtype=torch.bfloat16)
    d = host_tensor_desc(t)
    assert d.data == t.data_ptr() and d.ndim == 4 and list(d.shape) == [2, 4, 5, 128]
    assert d.dtype == L.DTYPES["bf16"]
    with pytest.raises(ValueError):
        host_tensor_desc(t.transpose(1, 2))                      # not contiguous
    with pytest.raises(ValueError):
        host_tensor_desc(torch.zeros((2, 4), dtype=torch.int8))  # no such storage dtype
    with pytest.raises(ValueError):
        host_tensor_desc(torch.zeros((1, 1, 1, 1, 2)))           # rank 5
    with pytest.raises(ValueError):
        host_tensor_desc(np.zeros((2, 4)))                       # not a tensor


def test_host_buffer_call_rejects_a_null_handle_and_bad_stage_size(kvc_lib):
    # no handle: rejected before anything else (no GPU needed)
    st = kvc_lib.lib.kvc_prefill_suffix_host(None, 0, None, None, None, None, None, None, -1, None)
    assert kvc_lib.STATUS[st] == "KVC_ERR_NULL"
