"""Shared pieces of the GPU parity tests (no arithmetic of the method)."""
import numpy as np
import pytest
import torch

TOL = {"f64": 1e-12, "f32": 1e-5, "bf16": 2e-2}
TORCH = {"f64": torch.float64, "f32": torch.float32, "bf16": torch.bfloat16}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def to_np(t):
    """Exact float64 copy of a bf16 / f32 / f64 tensor."""
    return t.detach().to(torch.float64).cpu().numpy()


def storage_np(cache, layer=0):
    K, V, P = cache.storage(layer)
    return to_np(K), to_np(V), P.cpu().numpy()


def device_tensor(a, dtype):
    """Host float64 array -> CUDA tensor of the storage dtype (rounded by torch)."""
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(TORCH[dtype])
