"""The multi-rank path of the benchmark on CPU: two gloo ranks, one data path each.

Requests are independent, so ranks share no data; the only collectives are the
barrier and the max-over-ranks reduction of the step time.  The whole-job rate is
world * units / slowest rank's time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 2.0 + rank            # rank 1 is slower
    dist.barrier()
    slow = bench.slowest_rank_ms(ms, world, device="cpu")
    rate = bench.whole_job_rate(1000, world, slow)
    q.put((rank, slow, rate))
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
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
    for rank, slow, rate in res:
        assert slow == 3.0                         # max over ranks
        assert rate == pytest.approx(2 * 1000 / 3e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.slowest_rank_ms(1.5, 1) == 1.5
    assert bench.whole_job_rate(10, 1, 2.0) == pytest.approx(5000.0)
