"""GPU parity of the router (a0, a1): the route kernel against the oracle on
identical fp32 logits (bit-exact selection, counts; fp32 statistics within
1e-5), and the router-logit kernel against the exact product."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_02_gb300 import synth
from mixture_experts_ffn_02_gb300.binding import Layer
from oracle import moe_oracle as O
from moe_check import STAT_RTOL, assert_close, np64

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
    b = lay.bufs
    np.testing.assert_array_equal(b["topk_idx"].cpu().numpy(), ref["topk_idx"])
    np.testing.assert_array_equal(b["counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_allclose(np64(b["gates"]), ref["gates"], rtol=STAT_RTOL, atol=1e-7)
    np.testing.assert_allclose(np64(b["f"]), ref["f"], rtol=STAT_RTOL, atol=0)
    np.testing.assert_allclose(np64(b["p"]), ref["p"], rtol=STAT_RTOL, atol=1e-9)
    assert float(b["aux"][0]) == pytest.approx(ref["aux"], rel=STAT_RTOL)
    st = b["router_stats"].cpu().numpy().astype(np.float64)
    assert st[0] == pytest.approx(ref["z_loss"], rel=STAT_RTOL)
    assert st[1] == pytest.approx(ref["entropy"], rel=STAT_RTOL, abs=1e-7)
    assert (st[2], st[3], st[5], st[6]) == (ref["count_min"], ref["count_max"],
                                            ref["unused"], ref["T_real"])
    assert st[4] == pytest.approx(ref["count_cv"], rel=1e-6, abs=1e-7)


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
