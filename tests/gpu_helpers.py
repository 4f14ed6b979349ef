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
    """Stored keys and values as [B, H_kv, C, d_h] float64 and positions [B, C]; a paged
    pool is gathered through the block table (slots without a block read as 0)."""
    K, V, P = cache.storage(layer)
    K, V, P = to_np(K), to_np(V), P.cpu().numpy()
    c = cache.config
    if not c.block_rows:
        return K, V, P
    table, _ = cache.block_table()
    out = []
    for pool in (K, V):
        x = np.zeros((c.batch, c.heads_kv, table.shape[1] * c.block_rows, c.head_dim))
        for b in range(c.batch):
            for j, blk in enumerate(table[b]):
                if blk >= 0:
                    x[b, :, j * c.block_rows:(j + 1) * c.block_rows] = pool[blk]
        out.append(x[:, :, :c.capacity])
    return out[0], out[1], P


def device_tensor(a, dtype):
    """Host float64 array -> CUDA tensor of the storage dtype (rounded by torch)."""
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(TORCH[dtype])
