"""The debug build's device bounds checks (``build(debug=True)``, compiled
with MOE_DEBUG_BOUNDS), through the C ABI.

* On valid inputs the checking build gives the release build's results bit
  for bit and a clean status word.
* A row index planted in ``inv`` past the permuted rows makes moe_combine
  latch MOE_ERR_BOUNDS; that slot is skipped and every other token's output
  is unchanged.
* A segment table (row_offsets) planted past the row capacity makes the bf16
  and the MXFP8 gate/up GEMMs latch MOE_ERR_BOUNDS and store nothing.

The planted inputs are given to the checking library only: every kernel of
those calls reads the planted values through a check before any access.
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_02_gb300 import binding, synth
from mixture_experts_ffn_02_gb300.binding import Layer

pytestmark = pytest.mark.gpu

BOUNDS = 10     # MOE_ERR_BOUNDS


@pytest.fixture(scope="module")
def dlib():
    lib = binding.load(debug=True)
    assert lib.moe_debug_bounds() == 1
    assert binding.load(debug=False).moe_debug_bounds() == 0
    return lib


def _layer(s, lib, training, seed=0):
    inp = synth.make_inputs(s, seed=seed, with_grad=training)
    lay = Layer.create(s, training=training, lib=lib)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    return lay, dev


SHAPE = synth.MoEShape("dbg", T=500, d=256, E=8, k=2, H=256, n_shared=0, H_shared=0)


@pytest.mark.parametrize("s", [synth.shape(1), synth.scaled(synth.shape(2), T=700),
                               synth.scaled(synth.shape(3), T=900, T_real=800)])
def test_debug_build_matches_release_bit_for_bit(dlib, s):
    out = {}
    for name, lib in (("release", binding.load(debug=False)), ("debug", dlib)):
        lay, dev = _layer(s, lib, training=True)
        lay.forward()
        lay.backward(dev["dY"])
        torch.cuda.synchronize()
        assert lay.status() == 0, name
        out[name] = {"y": lay.bufs["y"].clone(),
                     **{n: v.clone() for n, v in lay.grads.items() if v is not None}}
    for n, v in out["release"].items():
        assert torch.equal(v, out["debug"][n]), n


def test_planted_inv_row_is_caught_and_skipped(dlib):
    lay, _ = _layer(SHAPE, dlib, training=False)
    lay.forward()
    torch.cuda.synchronize()
    assert lay.status() == 0
    y0 = lay.bufs["y"].clone()
    inv = lay.bufs["inv"]
    t, j = 7, 1
    R = lay.R_cap
    keep = int(inv[t * SHAPE.k + j])
    inv[t * SHAPE.k + j] = R + 100                  # past the permuted rows
    lay.combine()
    torch.cuda.synchronize()
    assert lay.status() == BOUNDS
    assert lay.status() == 0                        # read and cleared
    y = lay.bufs["y"]
    others = torch.ones(SHAPE.T, dtype=torch.bool, device=y.device)
    others[t] = False
    assert torch.equal(y[others], y0[others])
    # token t keeps only its other slot: g_0 out_perm[inv(t, 0)]
    r0 = int(inv[t * SHAPE.k])
    g0 = float(lay.bufs["gates"].view(-1)[t * SHAPE.k])
    ref = (torch.tensor(g0, dtype=torch.float32, device=y.device) *
           lay.bufs["out_perm"][r0].float()).to(torch.bfloat16)   # fp32 product, one rounding
    assert torch.equal(y[t], ref)
    inv[t * SHAPE.k + j] = keep
    lay.combine()
    torch.cuda.synchronize()
    assert lay.status() == 0 and torch.equal(lay.bufs["y"], y0)


def _plant_roff(lay):
    ro = lay.bufs["row_offsets"]
    keep = ro.clone()
    ro[-1] = lay.R_cap + 128                        # the last segment runs past R_cap
    return keep


def test_planted_segment_table_stops_the_gate_up_gemm(dlib):
    lay, _ = _layer(SHAPE, dlib, training=False)
    lay.forward()
    torch.cuda.synchronize()
    keep = _plant_roff(lay)
    lay.bufs["h"].fill_(3.0)
    lay.gate_up()
    torch.cuda.synchronize()
    assert lay.status() == BOUNDS
    assert bool((lay.bufs["h"] == 3.0).all())       # no tile ran
    lay.bufs["row_offsets"].copy_(keep)
    lay.forward()
    torch.cuda.synchronize()
    assert lay.status() == 0


def test_planted_segment_table_stops_the_mx_gate_up_gemm(dlib):
    lay, _ = _layer(SHAPE, dlib, training=False)
    lay.mx_alloc()
    lay.mx_quantize_weights()
    lay.mx_forward()
    torch.cuda.synchronize()
    assert lay.status() == 0
    keep = _plant_roff(lay)
    lay.mx["h_q"].fill_(0x5A)
    lay.mx_gate_up()
    torch.cuda.synchronize()
    assert lay.status() == BOUNDS
    assert bool((lay.mx["h_q"] == 0x5A).all())
    lay.bufs["row_offsets"].copy_(keep)
    lay.mx_forward()
    torch.cuda.synchronize()
    assert lay.status() == 0
