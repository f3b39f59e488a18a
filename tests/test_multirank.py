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


class _FakeLayer:
    """CPU stand-in for a Layer in the host-side test of the data-parallel
    exchange: route_partials / route_finalize follow the entry points'
    documented definitions on CPU tensors."""

    def __init__(self, counts, p, k):
        import types
        self.cfg = types.SimpleNamespace(E=len(counts), k=k)
        self.bufs = {"counts": torch.tensor(counts, dtype=torch.int32),
                     "p": torch.tensor(p, dtype=torch.float32),
                     "f": torch.zeros(len(counts)), "aux": torch.zeros(1)}

    def route_partials(self, sums):
        E, k = self.cfg.E, self.cfg.k
        tr = float(self.bufs["counts"].sum()) / k
        sums[:E] = self.bufs["counts"].double()
        sums[E:2 * E] = self.bufs["p"].double() * tr
        sums[2 * E] = tr

    def route_finalize(self, sums):
        E, k = self.cfg.E, self.cfg.k
        T = float(sums[2 * E])
        self.bufs["f"] = (sums[:E] / (k * T)).float()
        self.bufs["p"] = (sums[E:2 * E] / T).float()
        self.bufs["aux"] = (E * (sums[:E] / (k * T)) @ (sums[E:2 * E] / T)).float().reshape(1)


def _dp_rank(rank, world, port, out, L_parts, k):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    from oracle import moe_oracle as O
    from mixture_experts_ffn_02_gb300 import dp
    r = O.route(L_parts[rank], k)
    lay = _FakeLayer(r["counts"], r["p"], k)
    g = dp.global_routing_stats(lay, dist, average=True)
    out[rank] = (lay.bufs["f"].numpy(), lay.bufs["p"].numpy(), float(lay.bufs["aux"][0]),
                 g.t_real_local, g.t_real_global, g.coef_scale)
    dist.barrier()
    dist.destroy_process_group()


def test_data_parallel_routing_statistics_over_two_gloo_ranks():
    """Two ranks route different token sets; after the exchange both hold the
    statistics of the whole batch (the oracle's route on the union), and the
    backward coefficient scale is world * T_local / T_global."""
    import numpy as np
    from oracle import moe_oracle as O
    rng = np.random.default_rng(5)
    k, E = 2, 8
    L_parts = [rng.standard_normal((300, E)).astype(np.float32),
               rng.standard_normal((500, E)).astype(np.float32)]
    full = O.route(np.concatenate(L_parts), k)
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_dp_rank, args=(r, world, port, out, L_parts, k))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r, n in ((0, 300), (1, 500)):
        f, p_, aux, tl, tg, scale = out[r]
        np.testing.assert_allclose(f, full["f"], rtol=1e-6)
        np.testing.assert_allclose(p_, full["p"], rtol=1e-6)
        assert aux == pytest.approx(full["aux"], rel=1e-6)
        assert (tl, tg) == (n, 800) and scale == pytest.approx(2 * n / 800)
