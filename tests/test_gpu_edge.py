"""Edge cases of the whole layer (forward + backward through the C ABI)
against the oracle: a batch of PAD tokens only, a single expert, a single
token, the widest router (E = 256) and every token on one expert."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_02_gb300 import synth
from mixture_experts_ffn_02_gb300.binding import Layer
from oracle import moe_oracle as O
from moe_check import (AdoptStored, Checker, logit_error_bound, np64, padded_layout,
                       reconcile_selection, stored_from_layer)

pytestmark = pytest.mark.gpu


def _run(s, seed=0, bias=None, valid=None):
    inp = synth.make_inputs(s, seed=seed, with_grad=True)
    if bias is not None:
        inp["bias"] = bias
    if valid is not None:
        inp["valid"] = valid
    lay = Layer.create(s, training=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    lay.forward()
    lay.backward(dev["dY"])
    torch.cuda.synchronize()
    assert lay.status() == 0
    return inp, lay


def _check_against_oracle(s, inp, lay):
    L = O.router_logits(inp["x"], inp["Wr"])
    bias = None if inp["bias"] is None else inp["bias"].numpy().astype(np.float64)
    key = L + (0.0 if bias is None else bias)
    real = np.ones(s.T, bool) if inp["valid"] is None else inp["valid"].numpy() != 0
    sel, _ = reconcile_selection(lay.bufs["topk_idx"].cpu().numpy(), key,
                                 logit_error_bound(np64(inp["x"]), np64(inp["Wr"])), s.k, real)
    r = O.route_stats(O.softmax(L), sel, real, bool(s.norm_topk))
    r["logits"] = L
    np.testing.assert_array_equal(lay.bufs["topk_idx"].cpu().numpy(), r["topk_idx"])
    np.testing.assert_array_equal(lay.bufs["counts"].cpu().numpy(), r["counts"])
    y = O.experts_forward(inp["x"], r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"],
                          inp["Ws_gu"], inp["Ws_down"], inp["valid"])[0]
    rop = padded_layout(r["topk_idx"], s.E)[2]
    adopt = AdoptStored(stored_from_layer(lay, True), rop, s.k)
    yi = O.experts_forward(inp["x"], r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"],
                           inp["Ws_gu"], inp["Ws_down"], inp["valid"], rnd=adopt)[0]
    fwd = dict(r, real=real)
    bargs = (inp["x"], inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"], inp["Ws_down"], fwd,
             inp["dY"])
    ex = O.backward(*bargs, norm_topk=bool(s.norm_topk), aux_coef=s.aux_coef)
    idl = O.backward(*bargs, norm_topk=bool(s.norm_topk), aux_coef=s.aux_coef, rnd=adopt)
    chk = Checker()
    adopt.check(chk)
    if np.any(y):
        chk.layer("y", lay.bufs["y"], y, yi)
    names = ["d_logits", "dW_down", "dW_gu", "dx", "dWr"] + (
        ["dWs_down", "dWs_gu"] if s.n_shared else [])
    for n in names:
        if np.any(ex[n]):
            chk.layer(n, lay.grads[n], ex[n], idl[n])
        else:
            assert not lay.grads[n].float().abs().max().item(), n
    chk.done()
    return r


def test_all_pad_batch():
    """T_real = 0: nothing is routed or counted; every output and gradient
    is zero (and no kernel divides by zero)."""
    s = synth.scaled(synth.shape(1), T=300, T_real=0)
    valid = torch.zeros(300, dtype=torch.uint8)
    inp, lay = _run(s, valid=valid)
    assert (lay.bufs["topk_idx"] == -1).all() and (lay.bufs["counts"] == 0).all()
    assert float(lay.bufs["aux"][0]) == 0.0
    assert int(lay.bufs["row_offsets"][-1]) == 0
    for t in (lay.bufs["y"], lay.grads["dx"], lay.grads["dW_gu"], lay.grads["dW_down"],
              lay.grads["dWr"], lay.grads["d_logits"], lay.grads["dWs_gu"],
              lay.grads["dWs_down"]):
        assert not t.float().abs().max().item()


def test_single_expert():
    s = synth.MoEShape("one", T=500, d=128, E=1, k=1, H=256, n_shared=1, H_shared=128)
    inp, lay = _run(s)
    assert lay.bufs["gates"].eq(1.0).all()
    _check_against_oracle(s, inp, lay)


def test_single_token():
    s = synth.MoEShape("tok", T=1, d=256, E=8, k=2, H=384, n_shared=1, H_shared=128)
    inp, lay = _run(s)
    _check_against_oracle(s, inp, lay)


def test_widest_router():
    s = synth.MoEShape("wide", T=700, d=256, E=256, k=8, H=128, n_shared=0, H_shared=0)
    inp, lay = _run(s)
    _check_against_oracle(s, inp, lay)


def test_every_token_on_one_expert():
    """A selection bias that sends every token to expert 0 (top-1): one full
    segment, every other expert empty (their dW must be exactly zero)."""
    s = synth.MoEShape("skew", T=900, d=256, E=16, k=1, H=256, n_shared=0, H_shared=0)
    bias = torch.tensor([100.0] + [0.0] * 15, dtype=torch.float32)
    inp, lay = _run(s, bias=bias)
    assert (lay.bufs["topk_idx"] == 0).all()
    r = _check_against_oracle(s, inp, lay)
    assert int(r["counts"][0]) == 900
    assert not lay.grads["dW_gu"][1:].float().abs().max().item()


def test_bounded_wait_timeout_latches_status_and_context_survives():
    """The failure path of the GEMM kernels' bounded waits, made to run out
    on purpose without any fault: a wait on an mbarrier that nothing arrives
    on gives up after its limit (50 ms), latches MOE_ERR_TIMEOUT in the status
    word and the kernel returns; the next layer call on the same context runs
    normally and matches the oracle."""
    import ctypes
    import time
    from mixture_experts_ffn_02_gb300 import binding
    s = synth.shape(1)
    inp, lay = _run(s)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    rc = lay.lib.moe_selftest_wait_timeout(ctypes.c_void_p(lay.ws.data_ptr()), 50_000_000,
                                           stream)
    assert rc == 0
    assert lay.status() == 7            # MOE_ERR_TIMEOUT, read (and cleared) by the host
    assert time.perf_counter() - t0 >= 0.045
    assert lay.status() == 0
    lay.forward()
    lay.backward(inp["dY"].cuda())
    torch.cuda.synchronize()
    assert lay.status() == 0
    _check_against_oracle(s, inp, lay)
    assert lay.lib.moe_selftest_wait_timeout(ctypes.c_void_p(lay.ws.data_ptr()), 0,
                                             stream) == 2           # MOE_ERR_SHAPE
