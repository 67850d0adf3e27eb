"""Multi-process bench logic on CPU (gloo, world size 2): replicas report the
slowest rank's time, and the job throughput counts every rank's work."""
import os
import socket
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


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [12.5, 10.0][rank]                       # rank 0 is the slow one
    slowest = bench.max_over_ranks(ms)
    thr = bench.aggregate_throughput(1e9, 4, slowest, world)
    dist.barrier()
    q.put((rank, slowest, thr))
    dist.destroy_process_group()


def test_replicas_max_time_and_aggregate_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, thr in res:
        assert slowest == 12.5
        assert thr == pytest.approx(2 * 1e9 * 4 / 12.5e-3)


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.aggregate_throughput(10.0, 2, 1000.0, 1) == pytest.approx(20.0)
