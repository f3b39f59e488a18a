"""GPU parity of the expert path (a3-a6): the tcgen05 grouped gate/up GEMM
with the SwiGLU epilogue, the grouped down GEMM, the dense shared expert and
the combine, each against the oracle's fp64 SwiGLU on the same rows.  The
routing is a seeded synthetic choice, so these tests isolate the GEMMs."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_02_gb300 import synth
from mixture_experts_ffn_02_gb300.binding import Layer
from oracle import moe_oracle as O
from moe_check import AdoptStored, Checker, np64, padded_layout, stored_from_layer

pytestmark = pytest.mark.gpu

CASES = [
    # name, T, d, E, k, H, n_shared, H_shared, pad, skew
    ("tiny", 256, 64, 4, 2, 128, 1, 128, 0, 0.0),
    ("ragged", 1000, 256, 4, 2, 384, 1, 192, 0, 0.0),
    ("kochi_slice", 700, 1536, 4, 2, 3072, 1, 3072, 0, 0.0),
    ("qwen_pad", 2100, 512, 8, 2, 768, 0, 0, 200, 0.0),
    ("deepseek_skew", 900, 2048, 64, 6, 1408, 2, 1408, 0, 1.1),
    ("many_experts", 1200, 1024, 128, 8, 768, 0, 0, 0, 0.0),
    ("odd_hidden", 300, 192, 6, 3, 320, 1, 64, 17, 0.5),
]


def _setup(T, d, E, k, H, ns, Hs, pad, skew, seed=0, training=False):
    s = synth.MoEShape("x", T=T, d=d, E=E, k=k, H=H, n_shared=ns, H_shared=Hs)
    inp = synth.make_inputs(s, seed=seed)
    valid = None
    if pad:
        valid = torch.ones(T, dtype=torch.uint8)
        valid[T - pad:] = 0
    topk = synth.random_topk(T, E, k, seed=seed + 1, valid=valid, skew=skew)
    g = torch.rand(T, k, generator=torch.Generator().manual_seed(seed + 2)) + 0.1
    g = (g / g.sum(1, keepdim=True)).float()
    if valid is not None:
        g[valid == 0] = 0
    lay = Layer.create(s, training=training)
    dev = {k_: (v.cuda() if isinstance(v, torch.Tensor) else v) for k_, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], valid=None if valid is None else valid.cuda())
    lay.bufs.update(topk_idx=topk.cuda(), gates=g.cuda())
    return s, inp, valid, topk, g, lay


@pytest.mark.parametrize("pairs", [None, "0", "1"])
@pytest.mark.parametrize("name,T,d,E,k,H,ns,Hs,pad,skew", CASES)
def test_expert_gemms_and_combine(name, T, d, E, k, H, ns, Hs, pad, skew, pairs, monkeypatch):
    """Forward GEMMs and combine with the default kernel choice, and with
    every product forced onto single CTAs ("0") or CTA pairs ("1")."""
    if pairs is not None:
        monkeypatch.setenv("MOE_GEMM_CTA_PAIRS", pairs)
    s, inp, valid, topk, g, lay = _setup(T, d, E, k, H, ns, Hs, pad, skew, training=True)
    lay.permute()
    lay.gate_up()
    lay.down()
    lay.shared()
    lay.combine()
    torch.cuda.synchronize()
    assert lay.status() == 0

    offsets, row_offsets, row_of_pair, perm_padded = padded_layout(topk.numpy(), E)
    R = int(row_offsets[-1])
    x = np64(inp["x"])
    Wg, Wu = O.split_gu(np64(inp["W_gu"]))
    Wd = np64(inp["W_down"])
    h_ref = np.zeros((R, H)); a_ref = np.zeros((R, H)); b_ref = np.zeros((R, H))
    o_ref = np.zeros((R, d)); o_ideal = np.zeros((R, d))
    # the storage-rounded oracle continuing from the GPU's valid rounding
    # choices of h (moe_check.AdoptStored), per (slot, expert) group of rows
    adopt = AdoptStored(stored_from_layer(lay, False), row_of_pair, k)
    tk = topk.numpy()
    for j in range(k):
        for e in range(E):
            toks = np.nonzero(tk[:, j] == e)[0]
            if toks.size == 0:
                continue
            rows = row_of_pair[toks * k + j]
            out, a, b, h = O.swiglu_parts(x[toks], Wg[e], Wu[e], Wd[e])
            h_ref[rows], a_ref[rows], b_ref[rows], o_ref[rows] = h, a, b, out
            o_ideal[rows] = O.swiglu_parts(x[toks], Wg[e], Wu[e], Wd[e], adopt,
                                           dict(e=e, j=j, rows=toks))[0]
    bufs = lay.bufs
    chk = Checker()
    chk.close("h", bufs["h"][:R], h_ref)
    chk.close("a", bufs["ab"][:R, :H], a_ref)
    chk.close("b", bufs["ab"][:R, H:], b_ref)
    chk.layer("out_perm", bufs["out_perm"][:R], o_ref, o_ideal)
    pad_rows = torch.from_numpy(perm_padded < 0)
    assert (bufs["h"][:R].cpu()[pad_rows].float() == 0).all()
    assert (bufs["out_perm"][:R].cpu()[pad_rows].float() == 0).all()

    vnp = None if valid is None else valid.numpy()
    y_ref, _ = O.experts_forward(inp["x"], topk.numpy(), g.numpy(), inp["W_gu"],
                                 inp["W_down"], inp["Ws_gu"], inp["Ws_down"], vnp)
    y_ideal, _ = O.experts_forward(inp["x"], topk.numpy(), g.numpy(), inp["W_gu"],
                                   inp["W_down"], inp["Ws_gu"], inp["Ws_down"], vnp,
                                   rnd=adopt)
    if ns:
        sg, su = O.split_gu(np64(inp["Ws_gu"]))
        real_rows = np.arange(T) if vnp is None else np.nonzero(vnp != 0)[0]
        s_ref = np.zeros((T, d)); s_ideal = np.zeros((T, d))
        s_ref[real_rows], *_ = O.swiglu_parts(x[real_rows], sg, su, np64(inp["Ws_down"]))
        s_ideal[real_rows], *_ = O.swiglu_parts(x[real_rows], sg, su, np64(inp["Ws_down"]),
                                                adopt, dict(shared=True, rows=real_rows))
        chk.layer("s_out", bufs["s_out"], s_ref, s_ideal)
    chk.layer("y", bufs["y"], y_ref, y_ideal)
    adopt.check(chk)
    chk.done()
    if valid is not None:
        assert (bufs["y"].cpu()[valid == 0].float() == 0).all()


def test_gate_up_repeatable():
    """Two launches on the same inputs give identical bytes (no races)."""
    s, inp, valid, topk, g, lay = _setup(1000, 512, 8, 2, 768, 0, 0, 0, 0.0)
    lay.permute()
    lay.gate_up()
    R = int(lay.bufs["row_offsets"][-1])
    h1 = lay.bufs["h"][:R].clone()
    lay.bufs["h"].zero_()
    lay.gate_up()
    torch.cuda.synchronize()
    assert torch.equal(h1, lay.bufs["h"][:R])


@pytest.mark.parametrize("name,T,d,E,k,H,ns,Hs,pad,skew", [CASES[1], CASES[3], CASES[4]])
def test_expert_ffn_call(name, T, d, E, k, H, ns, Hs, pad, skew):
    """moe_expert_ffn (gate/up, down and the shared expert in one call) then
    moe_combine: y against the oracle, and h, out_perm, s_out bit for bit
    the same as from the three separate calls."""
    s, inp, valid, topk, g, lay = _setup(T, d, E, k, H, ns, Hs, pad, skew)
    lay.permute()
    lay.expert_ffn()
    lay.combine()
    torch.cuda.synchronize()
    assert lay.status() == 0
    R = int(lay.bufs["row_offsets"][-1])
    one = {n: lay.bufs[n][:R].clone() for n in ("h", "out_perm")}
    one["y"] = lay.bufs["y"].clone()
    if ns:
        one["s_out"] = lay.bufs["s_out"].clone()
    vnp = None if valid is None else valid.numpy()
    y_ref, _ = O.experts_forward(inp["x"], topk.numpy(), g.numpy(), inp["W_gu"],
                                 inp["W_down"], inp["Ws_gu"], inp["Ws_down"], vnp)
    R_ = int(lay.bufs["row_offsets"][-1])
    adopt = AdoptStored(stored_from_layer(lay, False), padded_layout(topk.numpy(), E)[2], k)
    y_ideal, _ = O.experts_forward(inp["x"], topk.numpy(), g.numpy(), inp["W_gu"],
                                   inp["W_down"], inp["Ws_gu"], inp["Ws_down"], vnp,
                                   rnd=adopt)
    chk = Checker()
    chk.layer("y", one["y"], y_ref, y_ideal)
    adopt.check(chk)
    chk.done()
    assert R_ == R
    for n in ("h", "out_perm", "y", "s_out"):
        if n in one:
            lay.bufs[n].fill_(3.0)
    lay.gate_up()
    lay.down()
    lay.shared()
    lay.combine()
    torch.cuda.synchronize()
    assert lay.status() == 0
    for n, v in one.items():
        cur = lay.bufs[n][:R] if n in ("h", "out_perm") else lay.bufs[n]
        assert torch.equal(cur, v), n
