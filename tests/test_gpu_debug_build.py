"""The debug build (libkvc_debug.so, compiled with KVC_DEBUG): device bounds checks
on every length and slot index a kernel derives, standing in for a memory
checker.  A failed check records bit 32 of the device error word and skips the
access -- no trap, no assert -- so kvc_check reports it and the context stays
usable.

* A length that the host checks never let through is planted in the device
  lengths (KVC_OPT_TEST_PLANT_LENGTH: capacity + 5 for sequence 0); a decode
  step on the separate-kernel path reads it.  kvc_check must report the error
  word with the slot bit of the append kernel and the debug bounds bit, and no
  stored byte may change except the other sequence's new row.
* The small-case parity suites run once more against the debug library.
Both run in child processes (the binding loads one library per process).
"""
import os
import subprocess
import sys

import pytest

from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PLANT = r'''
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import numpy as np, torch
from kv_cache_append_rope_gb300 import _lib as L, workloads as W
from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
from gpu_helpers import device_tensor, raw_storage_np
assert L.VARIANT == "debug"
B, H, C, D = 2, 4, 128, 128
kd = device_tensor(W.normal_np((B, H, 32, D), 1), "bf16")
vd = device_tensor(W.normal_np((B, H, 32, D), 2), "bf16")
qd = device_tensor(W.normal_np((B, H, 32, D), 3), "bf16")
cache = KVCache(B, H, C, D)
cache.prefill_suffix(0, None, kd[:, :, :20].contiguous(), vd[:, :, :20].contiguous(), seqlen=[10, 20], out=False)
cache.set_option(L.OPT_DECODE_FUSED, 0)       # the separate-kernel step reads the device lengths
before = raw_storage_np(cache)
cache.set_option(L.OPT_TEST_PLANT_LENGTH, C + 5)
one = lambda x: x[:, :, 20:21].contiguous()
cache.append_attend(0, one(qd), one(kd), one(vd))   # host mirrors are sound: the call is enqueued
try:
    cache.check()
    print("NO ERROR REPORTED")
    sys.exit(1)
except KVCError as e:
    assert e.name == "KVC_ERR_DEVICE", e
    word = int(str(e).split("error word 0x")[1].split()[0], 16)
    print("error word", hex(word))
    assert word & 32 and word & 1, hex(word)
after = raw_storage_np(cache)
# sequence 1 appended its row at slot 20; nothing else changed (no write at slot C + 5 of
# sequence 0, which would land in the next head's rows)
for a, b in zip(before[:2], after[:2]):
    diff = np.argwhere(a != b)
    assert all(int(x[0]) == 1 and int(x[2]) == 20 for x in diff), diff[:5]
assert before[2][0].tolist() == after[2][0].tolist()
cache.reset()
cache.set_option(L.OPT_DECODE_FUSED, 1)
cache.append_attend(0, one(qd), one(kd), one(vd))
cache.check()
print("PLANT OK")
'''


def _child(code_or_args, timeout):
    env = dict(os.environ, KVC_LIB="debug")
    cmd = [sys.executable] + code_or_args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_planted_length_is_reported_without_an_out_of_range_access():
    need_gpu()
    from kv_cache_append_rope_gb300 import build
    build.build()
    code = PLANT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = _child(["-c", code], timeout=300)
    assert r.returncode == 0 and "PLANT OK" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]


def test_release_build_refuses_the_plant_option():
    need_gpu()
    from kv_cache_append_rope_gb300 import _lib as L
    from kv_cache_append_rope_gb300.kvc import KVCache, KVCError
    if L.VARIANT == "debug":
        pytest.skip("this process runs the debug build")
    cache = KVCache(1, 2, 8, 128)
    with pytest.raises(KVCError) as e:
        cache.set_option(L.OPT_TEST_PLANT_LENGTH, 20)
    assert e.value.name == "KVC_ERR_CONFIG"


def test_small_parity_suites_pass_on_the_debug_build():
    need_gpu()
    from kv_cache_append_rope_gb300 import _lib as L
    if L.VARIANT == "debug":
        pytest.skip("already running on the debug build")
    suites = ["tests/test_gpu_decode.py", "tests/test_gpu_prefix.py", "tests/test_gpu_window.py",
              "tests/test_gpu_paged.py", "tests/test_gpu_edges.py", "tests/test_gpu_read_rows.py",
              "tests/test_gpu_session.py"]
    r = _child(["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider"] + suites, timeout=1500)
    tail = r.stdout[-3000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
