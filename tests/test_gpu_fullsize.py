"""GPU parity at the full workload sizes, in the launch sequence bench.py
times (Layer.step: the fused router + route, the permute, the grouped GEMMs,
the combine folded into the shared expert's down GEMM where there is one,
and the backward), on outputs the oracle can compute one by one.

Checked in full: router logits, the routing (selection, counts; f, p, aux
and the metrics at 1e-5 against the oracle's route on the same fp32 logits),
the dispatch (offsets, padded row offsets, perm, inv) and the copied rows.
Checked on samples: the layer output y and the input gradient dx and logit
gradient of 48 seeded tokens; 16 columns of dW_down and 16 hidden units
(gate and up rows) of dW_gu for one expert, over all of that expert's rows;
the same for the shared expert.  dW_r is checked through the identity
dW_r = x^T d_logits, which holds at any size.
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_02_gb300 import synth
from mixture_experts_ffn_02_gb300.binding import Layer
from oracle import moe_oracle as O
from moe_check import (AdoptStored, Checker, assert_route_matches, logit_error_bound, np64,
                       padded_layout, reconcile_selection, route_on_gpu_logits,
                       stored_from_layer)

pytestmark = pytest.mark.gpu

N_TOK = 48
N_COL = 16


def run_bench_sequence(s):
    """The calls bench.py times for one step, on the full workload."""
    inp = synth.make_inputs(s, seed=0, with_grad=True)
    lay = Layer.create(s, training=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    lay.step(dev["dY"])           # bench.py's step: the same calls, in the same order
    torch.cuda.synchronize()
    assert lay.status() == 0
    return inp, lay


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_full_size_layer(cfg):
    s = synth.shape(cfg)
    inp, lay = run_bench_sequence(s)
    b, g = lay.bufs, lay.grads
    x = np64(inp["x"])
    Wr = np64(inp["Wr"])
    chk = Checker()

    # ---- router logits and routing, in full
    L = O.router_logits(inp["x"], inp["Wr"])
    chk.close("logits", b["logits"], L, tol=1e-5)
    bias = None if inp["bias"] is None else inp["bias"].numpy().astype(np.float64)
    key = L + (0.0 if bias is None else bias)
    real = np.ones(s.T, bool) if inp["valid"] is None else inp["valid"].numpy() != 0
    sel, adopted = reconcile_selection(b["topk_idx"].cpu().numpy(), key,
                                       logit_error_bound(x, Wr), s.k, real)
    probs = O.softmax(L)
    r = O.route_stats(probs, sel, real, bool(s.norm_topk))
    np.testing.assert_array_equal(b["topk_idx"].cpu().numpy(), r["topk_idx"])
    np.testing.assert_array_equal(b["counts"].cpu().numpy(), r["counts"])
    # the statistics and metrics at 1e-5: the oracle's route on the GPU's own
    # fp32 logits (the same keys, so the same selection bit for bit)
    assert_route_matches(b, route_on_gpu_logits(b, inp, s.k, s.norm_topk))

    # ---- dispatch, in full
    offsets, row_offsets, row_of_pair, perm_padded = padded_layout(r["topk_idx"], s.E)
    R = int(row_offsets[-1])
    np.testing.assert_array_equal(b["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(b["row_offsets"].cpu().numpy(), row_offsets)
    np.testing.assert_array_equal(b["inv"].cpu().numpy(), row_of_pair)
    np.testing.assert_array_equal(b["perm"][:R].cpu().numpy(), perm_padded)
    rows = torch.from_numpy(np.nonzero(perm_padded >= 0)[0]).cuda()
    toks = torch.from_numpy(perm_padded[perm_padded >= 0] // s.k).cuda()
    assert torch.equal(b["x_perm"][rows], lay.bufs["x"][toks])
    assert not b["x_perm"][:R][torch.from_numpy(perm_padded < 0).cuda()].any()

    # ---- sampled tokens: y, dx, d_logits
    rng = np.random.default_rng(cfg)
    ts = np.sort(rng.choice(s.T, size=min(N_TOK, s.T), replace=False))
    if not real.all():
        ts = np.unique(np.concatenate([ts, np.nonzero(~real)[0][:4]]))
    sub_real = real[ts]
    tsc = torch.from_numpy(ts)
    tsd = tsc.cuda()
    fwd = dict(topk_idx=r["topk_idx"][ts], gates=r["gates"][ts], probs=probs[ts],
               real=sub_real, f=r["f"])
    xs = inp["x"][tsc]
    # the storage-rounded oracle, continuing from the GPU's stored values
    # where they are the other valid rounding (moe_check.AdoptStored)
    stored = stored_from_layer(lay, True)
    adopt = AdoptStored(stored, row_of_pair, s.k, tokens=ts)
    for name, rnd in (("exact", None), ("ideal", adopt)):
        y_s, _ = O.experts_forward(xs, fwd["topk_idx"], fwd["gates"], inp["W_gu"],
                                   inp["W_down"], inp["Ws_gu"], inp["Ws_down"],
                                   sub_real.astype(np.uint8), rnd=rnd)
        fwd["y_" + name] = y_s
    chk.layer("y[sample]", b["y"][tsd], fwd["y_exact"], fwd["y_ideal"])
    # the aux term scales with 1/T_real of the whole batch, not of the sample
    coef = s.aux_coef * max(int(sub_real.sum()), 1) / int(real.sum())
    args = (xs, inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"], inp["Ws_down"], fwd,
            inp["dY"][tsc])
    ex = O.backward(*args, norm_topk=bool(s.norm_topk), aux_coef=coef)
    idl = O.backward(*args, norm_topk=bool(s.norm_topk), aux_coef=coef, rnd=adopt)
    chk.layer("dx[sample]", g["dx"][tsd], ex["dx"], idl["dx"])
    chk.layer("d_logits[sample]", g["d_logits"][tsd], ex["d_logits"], idl["d_logits"])
    adopt.check(chk)

    # ---- one expert's weight gradients on sampled columns / hidden units:
    # the expert's rows in segment order, the same products as the oracle's
    # backward (storage points through the same hook)
    counts = r["counts"]
    e = int(np.argsort(counts)[len(counts) // 2])
    seg = O.permute(r["topk_idx"], s.E)[1][offsets[e]:offsets[e + 1]]
    tok, slot = seg // s.k, seg % s.k
    gate = r["gates"][tok, slot]
    Wg, Wu = O.split_gu(np64(inp["W_gu"][e]))
    Wd = np64(inp["W_down"][e])
    dY = np64(inp["dY"])
    J = np.sort(rng.choice(s.H, size=N_COL, replace=False))
    adopt_e = AdoptStored(stored_from_layer(lay, True, cols=J), row_of_pair, s.k)
    res = {}
    for name, rnd in (("exact", None), ("ideal", adopt_e)):
        xe = x[tok]
        dWd = np.zeros((s.d, N_COL)); dWg = np.zeros((N_COL, s.d)); dWu = np.zeros((N_COL, s.d))
        for j in range(s.k):                       # the oracle's groups: (expert, slot)
            m = slot == j
            if not m.any():
                continue
            where = dict(e=e, j=j, rows=tok[m])
            _, a, bb, h = O.swiglu_parts(xe[m], Wg[J], Wu[J], Wd[:, J], rnd, where)
            d_out = O.stored_d_out(gate[m], dY[tok[m]], rnd, where)
            da, db = O.stored_swiglu_backward(d_out @ Wd[:, J], a, bb, rnd, where)
            dWd += d_out.T @ h                       # dW_down[e][:, J]
            dWg += da.T @ xe[m]                      # dW_gu[e][J, :]
            dWu += db.T @ xe[m]                      # dW_gu[e][H+J, :]
        res[name] = (dWd, dWg, dWu)
    gWd = g["dW_down"][e][:, torch.from_numpy(J).cuda()]
    gWg = g["dW_gu"][e][torch.from_numpy(J).cuda()]
    gWu = g["dW_gu"][e][torch.from_numpy(J + s.H).cuda()]
    for nm, gv, k_ in (("dW_down[e]", gWd, 0), ("dW_gate[e]", gWg, 1), ("dW_up[e]", gWu, 2)):
        chk.layer(nm, gv, res["exact"][k_], res["ideal"][k_])
    adopt_e.check(chk)

    if s.n_shared:
        Hs = s.Hs_total
        Js = np.sort(rng.choice(Hs, size=N_COL, replace=False))
        sg, su = O.split_gu(np64(inp["Ws_gu"]))
        Sd = np64(inp["Ws_down"])
        rows = np.nonzero(real)[0]
        xr, dYr = x[rows], dY[rows]
        adopt_s = AdoptStored(stored_from_layer(lay, True, shared_cols=Js), row_of_pair, s.k)
        res = {}
        for name, rnd in (("exact", None), ("ideal", adopt_s)):
            where = dict(shared=True, rows=rows)
            _, a, bb, h = O.swiglu_parts(xr, sg[Js], su[Js], Sd[:, Js], rnd, where)
            da, db = O.stored_swiglu_backward(dYr @ Sd[:, Js], a, bb, rnd, where)
            res[name] = (dYr.T @ h, da.T @ xr, db.T @ xr)
        jt = torch.from_numpy(Js).cuda()
        for nm, gv, k_ in (("dWs_down", g["dWs_down"][:, jt], 0),
                           ("dWs_gate", g["dWs_gu"][jt], 1),
                           ("dWs_up", g["dWs_gu"][jt + Hs], 2)):
            chk.layer(nm, gv, res["exact"][k_], res["ideal"][k_])
        adopt_s.check(chk)

    # ---- dW_r = x^T d_logits (identity at any size)
    dWr_id = x.T @ np64(g["d_logits"])
    chk.close("dWr=x^T.dL", g["dWr"], dWr_id, tol=1e-4)
    chk.done()
    del lay
    torch.cuda.empty_cache()
