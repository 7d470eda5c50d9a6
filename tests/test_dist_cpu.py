"""The multi-process reporting path of bench.py on CPU: gloo, world size 2.

bench.py runs one replica of the workload per GPU; the reported time is the
max over ranks and the reported work the sum over ranks.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    d = bench.Dist()
    d.init("gloo")
    t, u = bench.aggregate(d, local_seconds=1.0 + rank, local_units=10.0 * (rank + 1))
    d.barrier()
    out[rank] = (t, u)
    d.finish()


def test_aggregate_max_time_sum_units_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == (2.0, 30.0) and out[1] == (2.0, 30.0)


def test_single_process_aggregate_is_identity():
    import bench

    d = bench.Dist()
    assert bench.aggregate(d, 3.5, 7) == (3.5, 7)


def test_bench_refuses_a_world_size_other_than_gpus():
    """--gpus N under a launcher that started a different number of ranks is an error."""
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--steps", "1"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "WORLD_SIZE" in r.stderr
