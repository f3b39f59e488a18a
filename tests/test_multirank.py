"""The N > 1 path of bench.py on CPU: independent replicas, one process per
rank, timing = max over ranks, value = all ranks' tokens / that time.  Run
as two gloo ranks (world_size 2) on 127.0.0.1; no GPU, no data-path
collective beyond the timing reduction."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    ms_local = 100.0 + 50.0 * rank            # rank 1 is the slow one
    ms_max, value = bench.aggregate_ranks(ms_local, tokens_per_step=1000, steps=10,
                                          world=world, dist=dist)
    out[rank] = (ms_max, value)
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_sum_tokens():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        ms_max, value = out[r]
        assert ms_max == pytest.approx(150.0)
        assert value == pytest.approx(1000 * 10 * 2 / 0.150)


def test_single_rank_needs_no_process_group():
    import bench
    ms, v = bench.aggregate_ranks(200.0, 32768, 5, 1)
    assert ms == 200.0 and v == pytest.approx(32768 * 5 / 0.2)
