"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

Under torchrun each rank runs the whole workload on its own GPU (replicas,
no data-path collective); the job's throughput is the units all ranks
processed divided by the slowest rank's time.  These tests run that
aggregation, and the reference arm's rank-0-only rule, as two CPU processes.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, elapsed, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    value, t = bench.aggregate(1000.0, elapsed[rank], world)
    q.put((rank, value, t))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_aggregate_takes_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    elapsed = [2.0, 5.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, elapsed, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, value, t in res:
        assert t == 5.0
        assert value == pytest.approx(1000.0 * 2 / 5.0)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
