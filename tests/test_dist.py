"""Multi-rank host logic of bench.py on two CPU ranks (gloo): the slowest
rank's time is what every rank reports, and the job's throughput counts
every rank's replica of the workload (weak scaling).  No GPU involved."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = [2.0, 3.5][rank]
        slowest = bench.max_over_ranks(local_ms)
        value = bench.job_tflops(1e12, slowest, world)
        q.put((rank, slowest, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, slowest, value in got:
        assert slowest == 3.5                      # the slower rank's time
        # 2 ranks x 1 TFLOP over 3.5 ms
        assert value == pytest.approx(2 * 1e12 / 3.5e-3 / 1e12)


def test_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.job_tflops(4e12, 2.0, 1) == pytest.approx(2000.0)
