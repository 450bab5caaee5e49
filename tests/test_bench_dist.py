"""The multi-rank bench arithmetic on CPU: two `gloo` ranks, each with its own
timed-region length, agree on the slowest rank's time, and the job's tokens/s
counts every rank's tokens over that time (replicas of the layer, weak
scaling, no collective on the data path)."""
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_s = [2.0, 3.5][rank]
        t = bench.reduce_max(local_s, "cpu")
        v = bench.job_throughput(100 * 8, t, world)
        q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_job_throughput():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, v in res:
        assert t == pytest.approx(3.5)
        assert v == pytest.approx(2 * 800 / 3.5)


def test_single_process_without_a_group():
    import bench
    assert bench.reduce_max(1.25, "cpu") == 1.25
    assert bench.job_throughput(64, 2.0, 1) == 32.0
