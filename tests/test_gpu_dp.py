"""GPU parity of the data-parallel exchange kernels (moe_route_partials and
moe_route_finalize): a batch routed as two halves, with the halves' sums
added as an all-reduce would, gives the statistics of the whole batch; and
the backward with the global statistics and the scaled coefficient gives
each half's rows of the whole-batch logit gradient."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_02_gb300 import synth
from mixture_experts_ffn_02_gb300.binding import Layer
from oracle import moe_oracle as O
from moe_check import STAT_RTOL, assert_close, np64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [1, 3, 5])
def test_two_halves_give_the_whole_batch(cfg):
    s = synth.shape(cfg)
    T = 1200 if cfg != 1 else 256
    halves = [T // 3, T - T // 3]
    layers, sums, inps, refs = [], [], [], []
    for h, n in enumerate(halves):
        sh = synth.scaled(s, T=n, T_real=None)
        inp = synth.make_inputs(sh, seed=10 + h, with_grad=True)
        lay = Layer.create(sh, training=True)
        dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                       dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
        Lsyn = synth.random_logits(n, s.E, seed=20 + h)      # the same input to both sides
        lay.bufs["logits"] = Lsyn.cuda()
        lay.route()
        refs.append(Lsyn.numpy())
        sm = torch.empty(2 * s.E + 1, dtype=torch.float64, device="cuda")
        lay.route_partials(sm)
        layers.append(lay); sums.append(sm); inps.append(inp)
    total = sums[0] + sums[1]                      # what the all-reduce adds
    for lay in layers:
        lay.route_finalize(total)
    torch.cuda.synchronize()
    # the whole batch, routed by the oracle on the same logits
    full = O.route(np.concatenate(refs), s.k, bias=None if inps[0]["bias"] is None
                   else inps[0]["bias"].numpy())
    for lay in layers:
        np.testing.assert_allclose(np64(lay.bufs["f"]), full["f"], rtol=STAT_RTOL)
        np.testing.assert_allclose(np64(lay.bufs["p"]), full["p"], rtol=1e-5, atol=1e-8)
        assert float(lay.bufs["aux"][0]) == pytest.approx(full["aux"], rel=1e-5)
    # backward of the whole-batch aux term on each half: dY = 0 isolates it
    Tg = float(total[2 * s.E])
    for h, lay in enumerate(layers):
        Tl = float(sums[h][2 * s.E])
        lay.cfg.aux_coef = s.aux_coef * Tl / Tg * 50.0
        lay.permute()
        lay.gate_up(); lay.down(); lay.shared(); lay.combine()
        lay.backward(torch.zeros_like(lay.bufs["x"]))
        torch.cuda.synchronize()
        assert lay.status() == 0
        Lh = refs[h].astype(np.float64)
        probs = O.softmax(Lh)
        real = np.ones(Lh.shape[0], bool)
        # (aux_coef E / T_global) s (f_global - sum f_global s) with T_global
        ref = O.aux_logit_grad(probs, full["f"], real, s.aux_coef * Tl / Tg * 50.0)
        assert_close("d_logits[aux, global]", lay.grads["d_logits"], ref, tol=1e-4)
