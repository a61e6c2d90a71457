"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each with its own timed region;
the reported region is the slowest rank's and the throughput counts every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank          # rank 1 is slower
    mx = bench._max_over_ranks(local_ms, dist, device="cpu")
    rate = bench.aggregate_rate(1000.0, 4, world, mx)
    q.put((rank, mx, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, rate in res:
        assert mx == 15.0                                   # the slowest rank's region
        assert rate == pytest.approx(2 * 4 * 1000.0 / 0.015)  # both ranks' units over that region
