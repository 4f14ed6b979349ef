"""Times the float64 oracle on the host cores, for bench.py's CPU baseline.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only bench.py's
``cpu_baseline`` leg and its ``--impl reference`` arm use it.

``Workers(n)`` starts ``n`` fresh interpreters (``python -m oracle.timing``),
each limited to one BLAS/OpenMP thread, so ``n`` oracle calls run side by side
on ``n`` cores.  The processes are exec'd, never forked from a process that
holds a CUDA context, so they may be started at any time.  ``Workers.run``
hands each worker one task (the arrays of one oracle call, written to an
``.npz`` file), waits for all of them and returns every worker's compute time
-- the seconds of the oracle call alone, measured inside the worker, without
the interpreter start or the file transfer.  A batch of tasks that run side by
side takes ``max(seconds)`` of wall time on the host cores.

Task kinds (the arrays an ``.npz`` holds):

* ``decode``: q [steps, G, d], k, v [1, L0 + steps, d], L0 --
  ``attention.decode_steps_reference`` of one (sequence, key/value head) lane;
* ``suffix``: q [1, S, d], k, v [1, T, d], T, cut, rows --
  ``attention.suffix_reference`` of sampled suffix rows of one (sequence, head).
"""
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ONE_THREAD = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}


def run_task(z):
    """Runs the oracle call of one task (a mapping of arrays); returns its seconds."""
    from oracle import attention as A
    kind = str(z["kind"])
    t0 = time.perf_counter()
    if kind == "decode":
        A.decode_steps_reference(z["q"], z["k"], z["v"], int(z["L0"]), 10000.0, "bf16")
    elif kind == "suffix":
        A.suffix_reference(z["q"], z["k"], z["v"], np.arange(int(z["T"])), int(z["cut"]), 10000.0, "bf16",
                           rows=z["rows"])
    else:
        raise ValueError(f"unknown task kind {kind!r}")
    return time.perf_counter() - t0


def serve():
    """Worker loop: each line on stdin names an .npz task; the reply is its seconds."""
    for line in sys.stdin:
        path = line.strip()
        if not path:
            break
        with np.load(path) as z:
            secs = run_task(z)
        sys.stdout.write(f"{secs!r}\n")
        sys.stdout.flush()


class Workers:
    """``n`` one-thread oracle processes on the host cores."""

    def __init__(self, n):
        env = dict(os.environ, **ONE_THREAD)
        env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
        self.procs = [subprocess.Popen([sys.executable, "-m", "oracle.timing"], cwd=ROOT, env=env,
                                       stdin=subprocess.PIPE, stdout=subprocess.PIPE, text=True)
                      for _ in range(n)]
        self.dir = tempfile.TemporaryDirectory()
        self.count = 0

    @property
    def n(self):
        return len(self.procs)

    def run(self, tasks):
        """Runs up to n tasks side by side (one per worker); returns their seconds."""
        if len(tasks) > self.n:
            raise ValueError("more tasks than workers")
        paths = []
        for t in tasks:
            self.count += 1
            path = os.path.join(self.dir.name, f"task{self.count}.npz")
            np.savez(path, **t)
            paths.append(path)
        for p, path in zip(self.procs, paths):
            p.stdin.write(path + "\n")
            p.stdin.flush()
        secs = []
        for p, path in zip(self.procs, paths):
            line = p.stdout.readline()
            if not line:
                raise RuntimeError("an oracle worker exited")
            secs.append(float(line))
            os.remove(path)
        return secs

    def close(self):
        for p in self.procs:
            try:
                p.stdin.write("\n")
                p.stdin.flush()
                p.stdin.close()
            except Exception:
                pass
        for p in self.procs:
            try:
                p.wait(timeout=10)
            except Exception:
                p.kill()
        self.procs = []
        self.dir.cleanup()


if __name__ == "__main__":
    serve()
