"""A device-side wait that runs out is reported, not hung on, and the GPU stays usable.

The stall is made with a flag that nothing sets (KVC_OPT_TEST_STALL: the producer
warp of the next decode step issues no loads), never with a fault: the consumer
warps' bounded mbarrier waits give up after about a second, the kernel records
the timeout in the handle's device error word and returns, and kvc_check turns
it into KVC_ERR_DEVICE."""
import time

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, device_tensor, need_gpu, to_np
from kv_cache_append_rope_gb300 import _lib as L
from kv_cache_append_rope_gb300 import workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
from oracle import attention as A

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (32, 1)])     # m16n8k16 and tensor-core decode kernels
def test_bounded_wait_gives_up_and_is_reported(Hq, Hkv):
    need_gpu()
    B, D, C, L0 = 1, 128, 256, 100
    k = device_tensor(W.normal_np((B, Hkv, L0 + 1, D), 101), "bf16")
    v = device_tensor(W.normal_np((B, Hkv, L0 + 1, D), 102), "bf16")
    q = device_tensor(W.normal_np((B, Hq, L0 + 1, D), 103), "bf16")
    one = lambda x: x[:, :, L0:L0 + 1].contiguous()
    stalled = KVCache(B, Hq, C, D, heads_kv=Hkv)
    stalled.prefill_suffix(0, None, k[:, :, :L0].contiguous(), v[:, :, :L0].contiguous(), out=False)
    stalled.check()
    stalled.set_option(L.OPT_TEST_STALL, 1)
    t0 = time.time()
    stalled.append_attend(0, one(q), one(k), one(v))          # enqueued; the kernel waits, then gives up
    with pytest.raises(KVCError) as e:
        stalled.check()
    elapsed = time.time() - t0
    assert e.value.name == "KVC_ERR_DEVICE"
    assert "timed out" in str(e.value)
    assert 0.5 < elapsed < 60.0
    # the context is intact: a new cache computes the same step correctly
    fresh = KVCache(B, Hq, C, D, heads_kv=Hkv)
    fresh.prefill_suffix(0, None, k[:, :, :L0].contiguous(), v[:, :, :L0].contiguous(), out=False)
    out = to_np(fresh.append_attend(0, one(q), one(k), one(v)))
    ref = A.decode_steps_reference(to_np(q)[0, :, L0][None], to_np(k)[0], to_np(v)[0], L0, 10000.0, "bf16")
    assert np.abs(out[0, :, 0] - ref[0]).max() <= TOL["bf16"]
    fresh.check()
    torch.cuda.synchronize()
