"""Data-parallel routing statistics across torch.distributed ranks.

"spark-gpt" README: the auxiliary statistic is computed over the whole
data-parallel batch -- hard counts are synchronised across ranks, and the
differentiable local proxy is scaled so that averaging the ranks' gradients
yields the global-batch gradient.

This module is plumbing: the per-rank sums and the global f, p and aux are
computed by the library's kernels (moe_route_partials, moe_route_finalize);
torch.distributed only adds the sums across ranks (one all-reduce of 2E+1
float64 values, the layer's single exchange step).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass
class GlobalRouting:
    t_real_local: float
    t_real_global: float
    coef_scale: float      # multiply aux_coef and z_coef by this for the backward


def global_routing_stats(lay, dist, group=None, average: bool = True) -> GlobalRouting:
    """Replace ``lay``'s f, p and aux (from moe_route on this rank's tokens)
    by their values over all ranks of ``group``.

    Returns the factor for the backward's aux_coef and z_coef: their
    gradients are means over the global batch, so each rank's tokens weigh
    T_real(rank) / T_real(global); with ``average`` (the ranks' gradients are
    averaged, as DDP does) the factor also carries the rank count.  Reading
    the two token counts back is the one host synchronisation of the step.
    """
    import torch
    E = lay.cfg.E
    sums = torch.empty(2 * E + 1, dtype=torch.float64, device=lay.bufs["counts"].device)
    lay.route_partials(sums)
    t_local = sums[2 * E].clone()
    dist.all_reduce(sums, group=group)
    lay.route_finalize(sums)
    t = torch.stack([t_local, sums[2 * E]]).cpu()
    tl, tg = float(t[0]), float(t[1])
    world = dist.get_world_size(group) if average else 1
    scale = (tl / tg) * world if tg > 0 else 0.0
    return GlobalRouting(t_real_local=tl, t_real_global=tg, coef_scale=scale)
