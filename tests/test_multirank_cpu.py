"""The multi-rank host logic of bench.py on CPU: world size 2 over gloo.

Each rank runs an independent replica (weak scaling); the only exchange is the
barrier around the timed region and the max over ranks of the elapsed time.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    elapsed = 10.0 + 5.0 * rank              # rank 1 is the slow one
    results[rank] = bench.max_over_ranks(elapsed, world)
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        assert dict(results) == {0: 15.0, 1: 15.0}


@pytest.mark.parametrize("rank", ["1"])
def test_reference_arm_runs_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=rank, WORLD_SIZE="2", LOCAL_RANK=rank)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
