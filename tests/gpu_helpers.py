"""Shared pieces of the GPU parity tests (no arithmetic of the method)."""
import numpy as np
import pytest
import torch

from gpu_helpers_cpu import REL_GUARD, rel_err  # noqa: F401  (re-export)

TOL = {"f64": 1e-12, "f32": 1e-5, "bf16": 2e-2}


def assert_close(got, ref, dtype, what=""):
    """The contract (max-abs TOL[dtype]) and, for bf16, the relative-error regression
    guard REL_GUARD on every output row (the last axis is the head dimension).
    Returns the max-abs error."""
    err = float(np.abs(np.asarray(got) - np.asarray(ref)).max())
    assert err <= TOL[dtype], (what, err)
    if dtype == "bf16":
        rel = rel_err(got, ref)
        assert rel <= REL_GUARD, (what, "relative error", rel)
    return err
TORCH = {"f64": torch.float64, "f32": torch.float32, "bf16": torch.bfloat16}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def to_np(t):
    """Exact float64 copy of a bf16 / f32 / f64 tensor."""
    return t.detach().to(torch.float64).cpu().numpy()


def storage_np(cache, layer=0):
    """Logical snapshot of one layer through kvc_read_rows: keys and values as
    [B, H_kv, C, d_h] float64 and positions [B, C]; rows at or past a sequence's
    length read as 0 (positions -1).  Paged storage is gathered by the library."""
    K, V, P = cache.read_rows(layer)
    return to_np(K), to_np(V), P.cpu().numpy()


def raw_storage_np(cache, layer=0):
    """Every byte of a contiguous layer's storage (rows past the lengths included):
    keys and values [B, H_kv, C, d_h] float64, positions [B, C]."""
    assert not cache.config.block_rows, "raw storage is read from contiguous caches only"
    K, V, P = cache.storage(layer)
    return to_np(K), to_np(V), P.cpu().numpy()


def device_tensor(a, dtype):
    """Host float64 array -> CUDA tensor of the storage dtype (rounded by torch)."""
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(TORCH[dtype])
