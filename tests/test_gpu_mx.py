"""GPU parity of the MXFP8 routed experts against the MX oracle
(``oracle/mx_oracle.py``), through the C ABI.

* Quantisation of the bf16 weights and of the permuted x rows: codes and
  scale bytes bit for bit (both sides quantise the same bf16 values, and the
  scaling by a power of two is exact in fp32 and fp64 alike).
* The layer output y with MX experts: max normalised error <= 1e-2 against
  the fp64 MX oracle, which quantises x, the weights and its own fp64 hidden
  h the same way.  The GPU quantises its fp32 h, so a code of h may differ
  where fp32 and fp64 fall on the two sides of a rounding boundary; such
  codes are one step apart and rare, which the hidden-code check bounds.
  The MX output differs from the bf16 layer's by several percent, so the
  tolerance separates the two paths.
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_02_gb300 import synth
from mixture_experts_ffn_02_gb300.binding import Layer
from oracle import moe_oracle as O
from oracle import mx_oracle as M
from moe_check import Checker, logit_error_bound, np64, reconcile_selection

pytestmark = pytest.mark.gpu

ATOM = 512


def sf_byte(r, kb):
    return (r % 32) * 16 + (r // 32) * 4 + kb


def unpack_rows(atoms, K, rows):
    """Scale atoms [rows/128][K/128][512] -> scale bytes [rows][K/32]."""
    a = atoms.reshape(-1, K // 128, ATOM)
    r = np.arange(rows)[:, None]
    kb = np.arange(K // 32)[None, :]
    return a[r // 128, kb // 4, sf_byte(r % 128, kb % 4)]


def unpack_w_gu(atoms, E, H, d):
    """W_gu scale atoms [E][2H/128][d/128][512] -> [E][2H][d/32]."""
    a = atoms.reshape(E, 2 * H // 128, d // 128, ATOM)
    n = np.arange(2 * H)
    kb = np.arange(d // 32)
    return a[:, n[:, None] // 128, kb[None, :] // 4, sf_byte(n[:, None] % 128, kb[None, :] % 4)]


def unpack_w_down(atoms, E, d, H):
    """W_down scale atoms [E][d/128][H/128][512] -> [E][d][H/32]."""
    a = atoms.reshape(E, d // 128, H // 128, ATOM)
    n = np.arange(d)
    kb = np.arange(H // 32)
    return a[:, n[:, None] // 128, kb[None, :] // 4, sf_byte(n[:, None] % 128, kb[None, :] % 4)]


def u8(t, n=None):
    a = t.cpu().numpy()
    return a if n is None else a[:n]


def mx_layer(s, seed=0):
    inp = synth.make_inputs(s, seed=seed, with_grad=False)
    lay = Layer.create(s, training=False)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    lay.mx_alloc()
    lay.mx_quantize_weights()
    lay.mx_forward()
    torch.cuda.synchronize()
    assert lay.status() == 0
    return inp, lay


def route_like_gpu(s, inp, lay, rows=None):
    """Oracle routing on exact logits; near-tie tokens may keep the GPU's
    equally valid choice.  ``rows``: a sample of tokens (None = all)."""
    x = np64(inp["x"]) if rows is None else np64(inp["x"])[rows]
    L = O.router_logits(x, inp["Wr"])
    bias = None if inp["bias"] is None else inp["bias"].numpy().astype(np.float64)
    key = L + (0.0 if bias is None else bias)
    bound = logit_error_bound(x, np64(inp["Wr"]))
    valid = None if inp["valid"] is None else inp["valid"].numpy()
    if rows is not None and valid is not None:
        valid = valid[rows]
    real = np.ones(x.shape[0], bool) if valid is None else valid != 0
    gtop = lay.bufs["topk_idx"].cpu().numpy()
    if rows is not None:
        gtop = gtop[rows]
    sel, _ = reconcile_selection(gtop, key, bound, s.k, real)
    r = O.route_stats(O.softmax(L), sel, real, bool(s.norm_topk))
    return r, x, valid


# cfg, tokens, overrides: the 64- and 128-expert shapes keep E, k, the bias
# and the shared experts but get smaller d and H, so that the fp64 quantiser
# of all their weights stays within seconds (the KochiLLM and packed shapes
# keep their full dimensions; the full-size test below covers KochiLLM's)
SCALED = [(2, 700, {}), (3, 3001, {}), (4, 900, dict(d=512, H=384, H_shared=384)),
          (5, 1300, dict(d=512, H=256))]


def scaled_shape(cfg, T, over=None):
    s = synth.shape(cfg)
    T_real = None if s.T_real is None else T - T // 12
    return synth.scaled(s, T=T, T_real=T_real, **(over or {}))


@pytest.mark.parametrize("cfg,T,over", SCALED)
def test_mx_quantisation_bit_exact(cfg, T, over):
    """Weight codes and scales, and the permuted x rows (real rows: the
    token's codes; pad rows: zero), equal the oracle's quantiser."""
    s = scaled_shape(cfg, T, over)
    inp, lay = mx_layer(s)
    E, d, H = s.E, s.d, s.H
    mx = lay.mx
    c_gu, s_gu = M.mx_quantize(np64(inp["W_gu"]))
    np.testing.assert_array_equal(u8(mx["W_gu_q"], E * 2 * H * d).reshape(E, 2 * H, d), c_gu)
    np.testing.assert_array_equal(unpack_w_gu(u8(mx["W_gu_s"], E * 2 * H * d // 32), E, H, d),
                                  s_gu)
    c_dn, s_dn = M.mx_quantize(np64(inp["W_down"]))
    np.testing.assert_array_equal(u8(mx["W_down_q"], E * d * H).reshape(E, d, H), c_dn)
    np.testing.assert_array_equal(unpack_w_down(u8(mx["W_down_s"], E * d * H // 32), E, d, H),
                                  s_dn)
    R = lay.R_cap
    xq = u8(mx["x_q"], R * d).reshape(R, d)
    xs = unpack_rows(u8(mx["x_s"], R * d // 32), d, R)
    c_x, s_x = M.mx_quantize(np64(inp["x"]))
    inv = lay.bufs["inv"].cpu().numpy().reshape(s.T, s.k)
    roff = lay.bufs["row_offsets"].cpu().numpy()
    t_idx, j_idx = np.nonzero(inv >= 0)
    rows = inv[t_idx, j_idx]
    np.testing.assert_array_equal(xq[rows], c_x[t_idx])
    np.testing.assert_array_equal(xs[rows], s_x[t_idx])
    used = np.zeros(R, bool)
    used[rows] = True
    pad = ~used[: roff[-1]]
    assert (xq[: roff[-1]][pad] == 0).all() and (xs[: roff[-1]][pad] == 0).all()
    if s.n_shared:
        # the shared expert's weights, and x in token order with PAD tokens and
        # the padding to 128 rows as zeros
        Hs, Tp = s.n_shared * s.H_shared, (s.T + 127) // 128 * 128
        c, sc = M.mx_quantize(np64(inp["Ws_gu"]))
        np.testing.assert_array_equal(u8(mx["Ws_gu_q"]).reshape(2 * Hs, d), c)
        np.testing.assert_array_equal(unpack_rows(u8(mx["Ws_gu_s"]), d, 2 * Hs), sc)
        c, sc = M.mx_quantize(np64(inp["Ws_down"]))
        np.testing.assert_array_equal(u8(mx["Ws_down_q"]).reshape(d, Hs), c)
        np.testing.assert_array_equal(unpack_rows(u8(mx["Ws_down_s"]), Hs, d), sc)
        xv = np64(inp["x"])
        if inp["valid"] is not None:
            xv = np.where((inp["valid"].numpy() != 0)[:, None], xv, 0.0)
        xv = np.concatenate([xv, np.zeros((Tp - s.T, d))])
        c, sc = M.mx_quantize(xv)
        np.testing.assert_array_equal(u8(mx["xt_q"]).reshape(Tp, d), c)
        np.testing.assert_array_equal(unpack_rows(u8(mx["xt_s"]), d, Tp), sc)


@pytest.mark.parametrize("cfg,T,over", SCALED)
def test_mx_forward_matches_oracle(cfg, T, over):
    s = scaled_shape(cfg, T, over)
    inp, lay = mx_layer(s)
    r, x, valid = route_like_gpu(s, inp, lay)
    np.testing.assert_array_equal(lay.bufs["topk_idx"].cpu().numpy(), r["topk_idx"])
    y_mx, _ = M.experts_forward_mx(x, r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"],
                                   inp["Ws_gu"], inp["Ws_down"], valid)
    y_bf, _ = O.experts_forward(x, r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"],
                                inp["Ws_gu"], inp["Ws_down"], valid)
    chk = Checker()
    chk.close("y_mx", lay.bufs["y"], y_mx)
    e_mx = chk.rows[-1][1]
    chk.done()
    # the bf16 layer's output is far outside the MX tolerance: the test
    # tells the two paths apart
    rms = np.sqrt(np.mean(y_bf ** 2))
    assert np.abs(y_mx - y_bf).max() / rms > 5 * max(e_mx, 1e-3)


def test_mx_hidden_codes_match_oracle():
    """h codes of the fused gate/up epilogue against the oracle's own h
    quantised: at most 0.1% differ, each by one code step of the same
    block scale, or the block scale differs by one where the block maximum
    sits on a power of two."""
    s = scaled_shape(2, 700)
    inp, lay = mx_layer(s)
    r, x, valid = route_like_gpu(s, inp, lay)
    np.testing.assert_array_equal(lay.bufs["topk_idx"].cpu().numpy(), r["topk_idx"])
    E, d, H, R = s.E, s.d, s.H, lay.R_cap
    hq = u8(lay.mx["h_q"], R * H).reshape(R, H)
    hs = unpack_rows(u8(lay.mx["h_s"], R * H // 32), H, R)
    inv = lay.bufs["inv"].cpu().numpy().reshape(s.T, s.k)
    xq = M.mx_roundtrip(x)
    Wq = M.mx_roundtrip(np64(inp["W_gu"]))
    n_diff = n_all = 0
    for e in range(E):
        t_idx, j_idx = np.nonzero(r["topk_idx"] == e)
        if t_idx.size == 0:
            continue
        a = xq[t_idx] @ Wq[e, :H].T
        b = xq[t_idx] @ Wq[e, H:].T
        c_ref, s_ref = M.mx_quantize(O.silu(a) * b)
        rows = inv[t_idx, j_idx]
        c_gpu, s_gpu = hq[rows], hs[rows]
        same_scale = np.repeat(s_gpu == s_ref, 32, axis=1)
        step = (c_gpu.astype(int) & 0x7F) - (c_ref.astype(int) & 0x7F)
        diff = c_gpu != c_ref
        assert (np.abs(step[diff & same_scale]) <= 1).all()
        assert (np.abs(s_gpu.astype(int) - s_ref.astype(int)) <= 1).all()
        n_diff += int(diff.sum())
        n_all += diff.size
    assert n_all > 0 and n_diff <= 1e-3 * n_all, (n_diff, n_all)


def test_mx_full_size_kochillm_sampled():
    """The KochiLLM-shaped layer at its full size (T = 32768): every weight
    code and scale bit for bit, and y on a sample of tokens against the MX
    oracle evaluated on those tokens alone."""
    s = synth.shape(2)
    inp, lay = mx_layer(s)
    E, d, H = s.E, s.d, s.H
    c_gu, s_gu = M.mx_quantize(np64(inp["W_gu"]))
    np.testing.assert_array_equal(u8(lay.mx["W_gu_q"], E * 2 * H * d).reshape(E, 2 * H, d),
                                  c_gu)
    np.testing.assert_array_equal(
        unpack_w_gu(u8(lay.mx["W_gu_s"], E * 2 * H * d // 32), E, H, d), s_gu)
    del c_gu, s_gu
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(s.T, size=48, replace=False))
    rows[-1] = s.T - 1
    r, x, valid = route_like_gpu(s, inp, lay, rows)
    np.testing.assert_array_equal(lay.bufs["topk_idx"].cpu().numpy()[rows], r["topk_idx"])
    y_mx, _ = M.experts_forward_mx(x, r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"],
                                   inp["Ws_gu"], inp["Ws_down"], valid)
    chk = Checker()
    chk.close("y_mx[sample]", lay.bufs["y"][rows], y_mx)
    chk.done()


def test_mx_forward_is_deterministic():
    s = scaled_shape(5, 1300, dict(d=512, H=256))
    _, lay = mx_layer(s)
    y0 = lay.bufs["y"].clone()
    lay.mx_forward()
    torch.cuda.synchronize()
    assert torch.equal(y0, lay.bufs["y"])


def test_mx_rejects_code_buffers_off_32_bytes():
    """The MX kernels store 32 bytes per thread: a code buffer or out_perm
    that is 16- but not 32-byte aligned is refused before any launch."""
    from mixture_experts_ffn_02_gb300 import binding
    s = scaled_shape(5, 1300, dict(d=512, H=256))
    _, lay = mx_layer(s)
    keep = lay.mx["h_q"]
    lay.mx["h_q"] = keep[16:]
    with pytest.raises(binding.MoEError) as ei:
        lay.mx_gate_up()
    assert ei.value.code == 3
    lay.mx["h_q"] = keep
    keep = lay.bufs["out_perm"]
    lay.bufs["out_perm"] = keep.view(-1)[4:]
    with pytest.raises(binding.MoEError) as ei:
        lay.mx_down()
    assert ei.value.code == 3
    lay.bufs["out_perm"] = keep
    lay.mx_forward()
    torch.cuda.synchronize()
    assert lay.status() == 0


@pytest.mark.parametrize("cfg,T,over", [(2, 700, {}), (4, 900, dict(d=512, H=384, H_shared=384))])
def test_mx_forward_equals_its_steps(cfg, T, over):
    """moe_mx_forward is its steps in order: moe_mx_shared_ffn (s_out) then
    moe_combine after the routed MX calls give the same y bit for bit."""
    s = scaled_shape(cfg, T, over)
    _, lay = mx_layer(s)
    y_fwd = lay.bufs["y"].clone()
    lay.router_route()
    lay.mx_permute()
    lay.mx_gate_up()
    lay.mx_down()
    lay.mx_shared()
    lay.combine()
    torch.cuda.synchronize()
    assert lay.status() == 0
    assert torch.equal(y_fwd, lay.bufs["y"])


@pytest.mark.parametrize("cfg,n_tok", [(3, 48), (4, 4), (5, 6)])
def test_mx_full_size_sampled(cfg, n_tok):
    """The packed, 64-expert and 128-expert layers at their full sizes, in
    the configuration bench.py times: y on a sample of tokens (the last one
    and, for the packed batch, PAD tokens included) against the MX oracle
    evaluated on those tokens with only the experts they chose, and the
    codes of the first and last of those experts' weights bit for bit."""
    s = synth.shape(cfg)
    inp, lay = mx_layer(s)
    rng = np.random.default_rng(11 + cfg)
    rows = np.sort(rng.choice(s.T - 1, size=n_tok - 1, replace=False))
    rows = np.append(rows, s.T - 1)
    r, x, valid = route_like_gpu(s, inp, lay, rows)
    np.testing.assert_array_equal(lay.bufs["topk_idx"].cpu().numpy()[rows], r["topk_idx"])
    topk = r["topk_idx"]
    used = np.unique(topk[topk >= 0])
    topk_c = np.where(topk >= 0, np.searchsorted(used, np.maximum(topk, 0)), -1)
    W_gu = inp["W_gu"][torch.from_numpy(used)]
    W_down = inp["W_down"][torch.from_numpy(used)]
    y_mx, _ = M.experts_forward_mx(x, topk_c, r["gates"], W_gu, W_down, inp["Ws_gu"],
                                   inp["Ws_down"], valid)
    chk = Checker()
    chk.close("y_mx[sample]", lay.bufs["y"][rows], y_mx)
    chk.done()
    E, d, H = s.E, s.d, s.H
    q_gpu = u8(lay.mx["W_gu_q"], E * 2 * H * d).reshape(E, 2 * H, d)
    for j in (0, len(used) - 1):
        c, _ = M.mx_quantize(np64(W_gu[j]))
        np.testing.assert_array_equal(q_gpu[used[j]], c)


def _mx_run(s, bias=None, valid=None):
    inp = synth.make_inputs(s, seed=0, with_grad=False)
    if bias is not None:
        inp["bias"] = bias
    if valid is not None:
        inp["valid"] = valid
    lay = Layer.create(s, training=False)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    lay.mx_alloc()
    lay.mx_quantize_weights()
    lay.mx_forward()
    torch.cuda.synchronize()
    assert lay.status() == 0
    return inp, lay


def test_mx_all_pad_batch():
    """T_real = 0: no routed rows (the MX GEMMs get no tiles), the shared
    expert sees zero codes, and y is exactly zero."""
    s = synth.MoEShape("pad", T=300, d=256, E=4, k=2, H=128, n_shared=1, H_shared=128,
                       T_real=0)
    _, lay = _mx_run(s, valid=torch.zeros(300, dtype=torch.uint8))
    assert int(lay.bufs["row_offsets"][-1]) == 0
    assert not lay.bufs["y"].float().abs().max().item()


@pytest.mark.parametrize("name,shape,bias", [
    ("single_token", dict(T=1, d=256, E=8, k=2, H=384, n_shared=1, H_shared=128), None),
    ("one_expert_full", dict(T=900, d=256, E=16, k=1, H=256, n_shared=0, H_shared=0),
     [100.0] + [0.0] * 15),
])
def test_mx_edge_shapes(name, shape, bias):
    """One token (one padded 128-row block per tensor), and every token on
    one expert (one full segment, every other expert empty)."""
    s = synth.MoEShape(name, **shape)
    b = None if bias is None else torch.tensor(bias, dtype=torch.float32)
    inp, lay = _mx_run(s, bias=b)
    r, x, valid = route_like_gpu(s, inp, lay)
    np.testing.assert_array_equal(lay.bufs["topk_idx"].cpu().numpy(), r["topk_idx"])
    y_mx, _ = M.experts_forward_mx(x, r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"],
                                   inp["Ws_gu"], inp["Ws_down"], valid)
    chk = Checker()
    chk.close("y_mx", lay.bufs["y"], y_mx)
    chk.done()
