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


# ---------------------------------------------------------------- context-parallel exchange

def _cp_worker(rank, world, port, q):
    """Rank r decodes round-robin shard r of a small causal workload (the oracle stands
    in for the GPU decode), then exchanges (O, LSE) with the product helper."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import numpy as np
        import mla_inputs as mi
        from oracle import mla_oracle as mo
        from token_mla_paged_gb300.cp import gather_states
        sw = mi.cp_shards_bf16(scale=1 / 256, num_shards=world)
        B, H = sw.full.batch, sw.full.num_heads
        rows = sw.full.total_q                      # query tokens of the unsharded batch
        O_sh, L_sh = mo.mla_decode_workload(sw.shards)
        mine = slice(rank * rows, (rank + 1) * rows)   # shard-major: shard r's (request, token) rows
        o_local = torch.from_numpy(O_sh[mine].astype(np.float32))
        l_local = torch.from_numpy(L_sh[mine].astype(np.float32))
        o_all, l_all = gather_states(o_local, l_local)
        q.put((rank, o_all.numpy().astype(np.float64), l_all.numpy().astype(np.float64),
               O_sh.reshape(world, rows, H, 512).astype(np.float32).astype(np.float64),
               L_sh.reshape(world, rows, H).astype(np.float32).astype(np.float64)))
    finally:
        dist.destroy_process_group()


def test_cp_exchange_gathers_shards_in_rank_order():
    """Two gloo ranks: the gathered states are every shard's, at index = shard, on
    every rank, and merging them gives the unsharded decode."""
    import numpy as np
    import mla_inputs as mi
    from oracle import mla_oracle as mo
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_cp_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    sw = mi.cp_shards_bf16(scale=1 / 256, num_shards=world)
    Ofull, Lfull = mo.mla_decode_workload(sw.full)
    H = sw.full.num_heads
    for rank, o_all, l_all, o_want, l_want in res:
        assert o_all.shape == (world, sw.full.total_q, H, 512)
        assert np.array_equal(o_all, o_want) and np.array_equal(l_all, l_want)
        Om, Lm = mo.merge_states(o_all.reshape(world, -1, 512), l_all.reshape(world, -1))
        # fp32 transport of the shard states: the merge equals the unsharded result
        # to float32 rounding
        assert np.abs(Om - Ofull.reshape(-1, 512)).max() < 1e-5
        assert np.abs(Lm - Lfull.reshape(-1)).max() < 1e-5
