"""The multi-GPU form of the step is replicas only: each rank runs its own batch
with no data exchange, and the job's throughput is all ranks' steps over the
slowest rank's time.  These tests run bench.py's aggregation on two gloo ranks
on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
    val = bench.replica_throughput(100, ms, world)
    q.put((rank, ms, val))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("times", [(250.0, 310.0), (410.0, 120.0)])
def test_two_gloo_ranks_take_the_slowest_rank(times):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    slow = max(times)
    for rank, ms, val in got:
        assert ms == slow
        assert val == pytest.approx(world * 100 / (slow / 1e3))


def test_single_rank_is_its_own_time():
    import bench
    assert bench.max_over_ranks(123.5, 1, None) == 123.5
    assert bench.replica_throughput(10, 1000.0, 1) == pytest.approx(10.0)

