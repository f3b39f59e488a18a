"""GPU parity of the router (a0, a1): the route kernel against the oracle on
identical fp32 logits (bit-exact selection, counts; fp32 statistics within
1e-5), and the router-logit kernel against the exact product."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_02_gb300 import synth
from mixture_experts_ffn_02_gb300.binding import Layer
from oracle import moe_oracle as O
from moe_check import (assert_close, assert_route_matches, logit_error_bound, np64,
                       reconcile_selection, route_on_gpu_logits)

pytestmark = pytest.mark.gpu

ROUTE_CASES = [
    # T, E, k, quantum, norm, pad_tail, bias
    (256, 4, 2, None, 1, 0, False),
    (1000, 4, 2, 0.25, 1, 0, False),       # frequent exact ties
    (777, 8, 2, None, 1, 100, False),      # PAD tail
    (513, 8, 2, 0.5, 0, 37, False),        # no renormalisation, ties, PAD
    (1024, 64, 6, None, 1, 0, True),       # selection bias (Zipf)
    (999, 64, 6, 0.125, 1, 0, True),
    (2048, 128, 8, None, 1, 0, False),
    (300, 128, 8, 0.25, 0, 10, False),
    (1, 4, 1, None, 1, 0, False),          # single token
    (65, 256, 32, None, 1, 0, False),      # widest supported
    (100, 6, 3, 0.5, 1, 0, False),         # E not a power of two
    (100, 24, 5, None, 1, 0, False),
]


def _shape(T, E, k):
    return synth.MoEShape("route", T=T, d=64, E=E, k=k, H=64, n_shared=0, H_shared=0)


@pytest.mark.parametrize("T,E,k,quantum,norm,pad,use_bias", ROUTE_CASES)
def test_route_bit_exact(T, E, k, quantum, norm, pad, use_bias):
    s = _shape(T, E, k)
    L = synth.random_logits(T, E, seed=T + E, quantum=quantum)
    bias = synth.selection_bias(synth.scaled(s, zipf_bias=1.1)) if use_bias else None
    valid = None
    if pad:
        valid = torch.ones(T, dtype=torch.uint8)
        valid[T - pad:] = 0
    lay = Layer.create(s, training=False, norm_topk=norm)
    lay.bufs.update(logits=L.cuda(), bias=None if bias is None else bias.cuda(),
                    valid=None if valid is None else valid.cuda())
    lay.route()
    torch.cuda.synchronize()
    assert lay.status() == 0
    ref = O.route(L.numpy(), k, bias=None if bias is None else bias.numpy(),
                  valid=None if valid is None else valid.numpy(), norm_topk=bool(norm))
    assert_route_matches(lay.bufs, ref)


def test_route_equal_logits_tie_rule():
    """Equal logits: experts 0..k-1 everywhere; f = 1/k there; p = 1/E; aux = 1."""
    T, E, k = 333, 8, 3
    lay = Layer.create(_shape(T, E, k))
    lay.bufs["logits"] = torch.zeros(T, E, device="cuda")
    lay.route()
    idx = lay.bufs["topk_idx"].cpu().numpy()
    assert (idx == np.arange(k)).all()
    assert float(lay.bufs["aux"][0]) == pytest.approx(1.0, rel=1e-6)
    np.testing.assert_allclose(lay.bufs["p"].cpu().numpy(), 1.0 / E, rtol=1e-6)


def test_route_nonfinite_sets_status():
    T, E, k = 64, 4, 2
    lay = Layer.create(_shape(T, E, k))
    L = torch.randn(T, E)
    L[5, 2] = float("nan")
    lay.bufs["logits"] = L.cuda()
    lay.route()
    assert lay.status() == 9          # MOE_ERR_NONFINITE
    assert lay.status() == 0          # reading clears it


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_router_logits_close_to_exact(cfg):
    s = synth.shape(cfg)
    s = synth.scaled(s, T=min(s.T, 3000), T_real=None)
    inp = synth.make_inputs(s, seed=7)
    lay = Layer.create(s)
    lay.bufs.update(x=inp["x"].cuda(), Wr=inp["Wr"].cuda())
    lay.router_logits()
    exact = O.router_logits(inp["x"], inp["Wr"])
    # fp32 accumulation over d terms
    assert_close("logits", lay.bufs["logits"], exact, tol=1e-5)


FUSED_CASES = [
    # d, E, k, T, pad, zipf, norm
    (64, 4, 2, 256, 0, 0.0, 1),
    (1536, 4, 2, 3001, 0, 0.0, 1),          # KochiLLM width, ragged tail of the 8-token tiles
    (512, 8, 2, 2049, 170, 0.0, 1),         # packed-batch width with a PAD tail
    (256, 16, 4, 1003, 0, 1.1, 0),          # selection bias, no renormalisation
    (128, 8, 8, 77, 5, 0.0, 1),             # k = E
    (64, 4, 1, 1, 0, 0.0, 1),               # single token
    (256, 64, 6, 500, 0, 1.1, 1),           # E > 16: the two-step path
    # several units per warp (each warp's two row buffers reused in turn)
    (1536, 4, 2, 20000, 0, 0.0, 1),
    (512, 8, 2, 40000, 300, 0.0, 1),
    (1024, 16, 2, 9000, 0, 1.1, 1),
]


@pytest.mark.parametrize("d,E,k,T,pad,zipf,norm", FUSED_CASES)
def test_router_route_matches_oracle(d, E, k, T, pad, zipf, norm):
    """moe_router_route (router and routing in one kernel for E <= 16)
    against the oracle on exact logits, with near-ties resolved by the fp32
    error bound; and against moe_route run on the logits it wrote, which
    must give the same selection, gates and statistics bit for bit."""
    s = synth.MoEShape("rr", T=T, d=d, E=E, k=k, H=64, n_shared=0, H_shared=0,
                       T_real=(T - pad) if pad else None, zipf_bias=zipf, norm_topk=norm)
    inp = synth.make_inputs(s, seed=d + E + T)
    lay = Layer.create(s)
    lay.bufs.update(x=inp["x"].cuda(), Wr=inp["Wr"].cuda(),
                    bias=None if inp["bias"] is None else inp["bias"].cuda(),
                    valid=None if inp["valid"] is None else inp["valid"].cuda())
    lay.router_route()
    torch.cuda.synchronize()
    assert lay.status() == 0
    b = {n: v.clone() for n, v in lay.bufs.items()
         if n in ("logits", "topk_idx", "gates", "counts", "f", "p", "aux", "router_stats")}

    L_exact = O.router_logits(inp["x"], inp["Wr"])
    assert_close("logits", b["logits"], L_exact, tol=1e-5)
    key = L_exact + (0.0 if inp["bias"] is None else inp["bias"].numpy().astype(np.float64))
    real = np.ones(T, bool) if inp["valid"] is None else inp["valid"].numpy() != 0
    sel, _ = reconcile_selection(b["topk_idx"].cpu().numpy(), key,
                                 logit_error_bound(np64(inp["x"]), np64(inp["Wr"])), k, real)
    r = O.route_stats(O.softmax(L_exact), sel, real, bool(norm))
    np.testing.assert_array_equal(b["topk_idx"].cpu().numpy(), r["topk_idx"])
    np.testing.assert_array_equal(b["counts"].cpu().numpy(), r["counts"])
    # the statistics at 1e-5: the oracle's route on the logits this call wrote
    assert_route_matches(b, route_on_gpu_logits(b, inp, k, norm))

    # the separate route kernel on the same fp32 logits: the same selection,
    # gates, counts, f, p and aux bit for bit (p is a sum of per-token fixed-
    # point integers, so it does not depend on how tokens were spread over
    # lanes and blocks); the count metrics exactly; the z-loss and entropy
    # means are fp32 sums whose order follows that spread
    lay.route()
    torch.cuda.synchronize()
    assert lay.status() == 0
    for n in ("topk_idx", "gates", "counts", "f", "p", "aux"):
        assert torch.equal(lay.bufs[n], b[n]), n
    st, st_f = lay.bufs["router_stats"].cpu(), b["router_stats"].cpu()
    assert torch.equal(st[2:], st_f[2:])
    np.testing.assert_allclose(st[:2].numpy(), st_f[:2].numpy(), rtol=1e-6, atol=1e-7)
