"""Host-side pieces of bench.py that need no GPU.

* The oracle workers (``oracle.timing.Workers``): one-thread interpreters that run
  oracle calls side by side and report each call's compute time; the result a
  worker computes is the oracle's own (the same call made here).
* The reference arm's input builder draws the same seeded tensors as the GPU arm
  without loading libkvc (checked in a fresh interpreter, on the CPU).
"""
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_oracle_workers_run_tasks_side_by_side():
    from oracle.timing import Workers, run_task
    rng = np.random.default_rng(0)
    L0, steps, G = 200, 4, 4
    dec = {"kind": "decode", "q": rng.standard_normal((steps, G, 128)), "k": rng.standard_normal((1, L0 + steps, 128)),
           "v": rng.standard_normal((1, L0 + steps, 128)), "L0": np.int64(L0)}
    T, cut = 400, 300
    suf = {"kind": "suffix", "q": rng.standard_normal((1, T - cut, 128)), "k": rng.standard_normal((1, T, 128)),
           "v": rng.standard_normal((1, T, 128)), "T": np.int64(T), "cut": np.int64(cut),
           "rows": np.arange(0, T - cut, 9)}
    w = Workers(2)
    try:
        secs = w.run([dec, suf])
        assert len(secs) == 2 and all(0.0 < s < 60.0 for s in secs)
        assert len(w.run([suf])) == 1
    finally:
        w.close()
    assert run_task(dec) > 0.0


def test_reference_inputs_do_not_load_the_library():
    code = (
        "import sys, torch\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "sys.argv = ['bench.py']\n"
        "import bench\n"
        "b = bench.make_bench('gqa_decode', torch.device('cpu'), batch=2, with_cache=False)\n"
        "tasks, work, desc = b.cpu_tasks(3, steps=2)\n"
        "assert len(tasks) == 3 and all(w > 0 for w in work)\n"
        "assert tasks[0]['q'].shape == (2, 4, 128) and tasks[0]['k'].shape[1] == int(tasks[0]['L0']) + 2\n"
        "cfg = b.config()\n"
        "assert cfg['workload'] == 'gqa_decode' and cfg['storage'] == 'contiguous'\n"
        "assert not any('libkvc' in m or m.endswith('._lib') for m in sys.modules), [m for m in sys.modules if 'kvc' in m]\n"
        "print('ok')\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_cpu_baseline_times_rounds_up_to_the_requested_seconds():
    """bench.cpu_baseline repeats rounds of one task per worker until the requested wall
    time and reports the rounds' work over the sum of each round's slowest task."""
    code = (
        "import sys, torch\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "sys.argv = ['bench.py']\n"
        "import bench\n"
        "from oracle.timing import Workers\n"
        "b = bench.make_bench('gqa_decode', torch.device('cpu'), batch=2, with_cache=False)\n"
        "bench.CPU_TASK['gqa_decode'] = dict(steps=1)\n"
        "w = Workers(2)\n"
        "try:\n"
        "    line = bench.cpu_baseline(b, w, 'GB/s', seconds=0.5)\n"
        "finally:\n"
        "    w.close()\n"
        "rounds = int(line['sample'].split()[0])\n"
        "assert line['cores'] == 2 and line['kind'] == 'oracle' and line['value'] > 0\n"
        "assert line['seconds'] >= 0.5 and rounds >= 1, line\n"
        "assert line['cpu_seconds'] >= line['seconds'] * 0.9, line\n"
        "assert line['one_core']['cores'] == 1 and line['one_core']['seconds'] >= 0.1, line\n"
        "print('ok')\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
