"""The benchmark's multi-rank logic on CPU: two gloo ranks, each timing its own replica of
the batch; the job's time is the slowest rank's and the value counts every rank's bytes."""
import os
import socket
import sys

import pytest

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 100.0 + 50.0 * rank              # rank 1 is the slow one
        total = bench.max_over_ranks(mine, dist, "cpu")
        value = bench.whole_job_gbps(2_000_000_000, 10, world, total)
        dist.barrier()
        q.put((rank, total, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_weak_scaling_value():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, total, value in got:
        assert total == 150.0                     # the slower rank's time, on both ranks
        assert value == pytest.approx(2 * 2e9 * 10 / 0.150 / 1e9)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_gbps(1e9, 4, 1, 1000.0) == pytest.approx(4.0)
