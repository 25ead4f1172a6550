"""The multi-replica path of bench.py on CPU: two gloo ranks (127.0.0.1), each with its own
timing, must both report the slowest rank's time, and the job's throughput counts every
rank's work over that time (independent replicas, weak scaling; no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 10.0 + 5.0 * rank                # rank 1 is the slower replica
        worst = bench.max_over_ranks(my_ms, "cpu")
        dist.barrier()
        q.put((rank, worst, bench.replica_throughput(1e12, 4, world, worst)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_report_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, tput in got:
        assert worst == 15.0
        assert tput == pytest.approx(1e12 * 4 * 2 / 0.015 / 1e12)


def test_single_process_needs_no_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.replica_throughput(2e12, 10, 1, 1000.0) == pytest.approx(20.0)
