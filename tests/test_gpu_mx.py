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
from moe_check import (AdoptStored, Checker, bf16_round, frob_err, logit_error_bound, np64,
                       padded_layout, reconcile_selection, stored_from_layer)

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


def unpack_w(atoms, E, N, K):
    """Per-expert scale atoms [E][N/128][K/128][512] of N rows quantised
    along K -> scale bytes [E][N][K/32]."""
    a = atoms.reshape(E, N // 128, K // 128, ATOM)
    n = np.arange(N)
    kb = np.arange(K // 32)
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


def check_mx_y(chk, name, lay, s, x, topk, gates, W_gu, W_down, Ws_gu, Ws_down, valid,
               tokens=None):
    """y of the MX forward against the MX oracle at the bounds of every bf16
    output: max-normalised |gpu - ideal| <= 1e-2, where ideal continues from
    the GPU's valid choices at its rounding points (the h codes and each
    routed slot's bf16 output), and Frobenius-relative |gpu - exact| <= 1e-2.
    ``tokens``: the oracle's rows are these tokens of the batch.  Returns the
    exact y."""
    row_of_pair = lay.bufs["inv"].cpu().numpy()
    adopt = AdoptStored(stored_from_layer(lay, False), row_of_pair, s.k, tokens=tokens)
    args = (x, topk, gates, W_gu, W_down, Ws_gu, Ws_down, valid)
    y_ex, _ = M.experts_forward_mx(*args)
    y_id, _ = M.experts_forward_mx(*args, rnd=adopt)
    gpu = lay.bufs["y"] if tokens is None else lay.bufs["y"][torch.from_numpy(tokens).cuda()]
    chk.layer(name, gpu, y_ex, y_id)
    adopt.check(chk)
    return y_ex


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
    y_bf, _ = O.experts_forward(x, r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"],
                                inp["Ws_gu"], inp["Ws_down"], valid)
    chk = Checker()
    y_mx = check_mx_y(chk, "y_mx", lay, s, x, r["topk_idx"], r["gates"], inp["W_gu"],
                      inp["W_down"], inp["Ws_gu"], inp["Ws_down"], valid)
    e_mx = chk.rows[0][1]                          # |gpu - ideal| max
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
    chk = Checker()
    check_mx_y(chk, "y_mx[sample]", lay, s, x, r["topk_idx"], r["gates"], inp["W_gu"],
               inp["W_down"], inp["Ws_gu"], inp["Ws_down"], valid, tokens=rows)
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
    lay.bufs["out_perm"] = keep.view(-1)[8:]          # 16 bytes in (bf16)
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
    chk = Checker()
    check_mx_y(chk, "y_mx[sample]", lay, s, x, topk_c, r["gates"], W_gu, W_down,
               inp["Ws_gu"], inp["Ws_down"], valid, tokens=rows)
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
    chk = Checker()
    check_mx_y(chk, "y_mx", lay, s, x, r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"],
               inp["Ws_gu"], inp["Ws_down"], valid)
    chk.done()


# --------------------------------------------------------------------------
# The MXFP8 training step: moe_mx_forward_train + moe_mx_backward
# --------------------------------------------------------------------------

def mx_train_layer(s, seed=0):
    inp = synth.make_inputs(s, seed=seed, with_grad=True)
    lay = Layer.create(s, training=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    lay.mx_alloc()
    lay.mx_quantize_weights()
    lay.mx_step(dev["dY"])
    torch.cuda.synchronize()
    assert lay.status() == 0
    return inp, lay


def train_fwd(s, inp, r):
    fwd = dict(r)
    fwd["real"] = np.ones(s.T, bool) if inp["valid"] is None else inp["valid"].numpy() != 0
    return fwd


def half_ulp_bf16_of(v):
    a = np.abs(v)
    return np.where(a > 0, np.exp2(np.floor(np.log2(np.where(a > 0, a, 1.0))) - 8), 0.0)


@pytest.mark.parametrize("cfg,T,over", SCALED)
def test_mx_train_operand_codes_bit_exact(cfg, T, over):
    """The data-gradient products' operands: each expert's W_gu^T and
    W_down^T quantised along 2H and d, bit for bit with the oracle's
    quantiser; the codes of d_out = g dY (along d) bit for bit with the
    oracle quantising the same fp32 products (the fp32 gate times the bf16
    dY, rounded to fp32 as one multiply does), pad rows zero; and the codes
    of d_gu (along 2H), quantised from fp32 values the GPU does not keep:
    each block scale is that of the stored bf16 d_gu or one less, and each
    code lies between the e4m3 roundings, under the GPU's scale, of the
    stored value minus and plus half a bf16 ulp (the fp32 value lies there,
    and the rounding is monotone)."""
    s = scaled_shape(cfg, T, over)
    inp, lay = mx_train_layer(s)
    E, d, H, R = s.E, s.d, s.H, lay.R_cap
    mx = lay.mx
    c, sc = M.mx_quantize(np.swapaxes(np64(inp["W_gu"]), 1, 2))           # [E][d][2H]
    np.testing.assert_array_equal(u8(mx["W_gu_tq"], E * d * 2 * H).reshape(E, d, 2 * H), c)
    np.testing.assert_array_equal(unpack_w(u8(mx["W_gu_ts"], E * d * 2 * H // 32), E, d,
                                           2 * H), sc)
    c, sc = M.mx_quantize(np.swapaxes(np64(inp["W_down"]), 1, 2))         # [E][H][d]
    np.testing.assert_array_equal(u8(mx["W_down_tq"], E * H * d).reshape(E, H, d), c)
    np.testing.assert_array_equal(unpack_w(u8(mx["W_down_ts"], E * H * d // 32), E, H, d), sc)
    inv = lay.bufs["inv"].cpu().numpy().reshape(-1)
    pair = np.nonzero(inv >= 0)[0]
    rows = inv[pair]
    gates = lay.bufs["gates"].cpu().numpy().reshape(-1)[pair].astype(np.float32)
    dY = inp["dY"].float().numpy()[pair // s.k]
    c, sc = M.mx_quantize((gates[:, None] * dY).astype(np.float64))   # fp32 products
    q = u8(mx["dout_q"], R * d).reshape(R, d)
    sb = unpack_rows(u8(mx["dout_s"], R * d // 32), d, R)
    np.testing.assert_array_equal(q[rows], c)
    np.testing.assert_array_equal(sb[rows], sc)
    used = np.zeros(R, bool)
    used[rows] = True
    n_rows = int(lay.bufs["row_offsets"][-1])
    pad = ~used[:n_rows]
    assert not q[:n_rows][pad].any() and not sb[:n_rows][pad].any()
    # d_gu
    K = 2 * H
    v = np64(lay.intermediates()["d_gu"])[rows]
    q = u8(mx["dgu_q"], R * K).reshape(R, K)[rows]
    sb = unpack_rows(u8(mx["dgu_s"], R * K // 32), K, R)[rows]
    _, s_bf = M.mx_quantize(v)
    assert np.isin(sb.astype(int) - s_bf.astype(int), (0, -1)).all()
    scale = np.repeat(np.exp2(sb.astype(np.float64) - 127.0), 32, axis=1)
    hu = half_ulp_bf16_of(v)
    lo = M.e4m3_decode(M.e4m3_round((v - hu) / scale))
    hi = M.e4m3_decode(M.e4m3_round((v + hu) / scale))
    got = M.e4m3_decode(q)
    assert ((got >= lo) & (got <= hi)).all()
    # and it is not the quantisation of the bf16 copy: that differs in a few
    # percent of the codes (about 2%), each by one e4m3 step
    c_bf, _ = M.mx_quantize(v)
    frac = float((c_bf != q).mean())
    assert 1e-3 < frac < 0.1, frac


@pytest.mark.parametrize("cfg,T,over", SCALED)
def test_mx_train_step_matches_oracle(cfg, T, over):
    """y and every gradient of the MXFP8 training step against the MX
    training oracle: max normalised |gpu - ideal| <= 1e-2, where ideal
    continues from the GPU's stored bf16 values where they are the other
    valid rounding, and Frobenius-relative |gpu - exact| <= 1e-2."""
    s = scaled_shape(cfg, T, over)
    inp, lay = mx_train_layer(s)
    r, x, valid = route_like_gpu(s, inp, lay)
    np.testing.assert_array_equal(lay.bufs["topk_idx"].cpu().numpy(), r["topk_idx"])
    fwd = train_fwd(s, inp, r)
    adopt = AdoptStored(stored_from_layer(lay, True), padded_layout(r["topk_idx"], s.E)[2], s.k)
    fw = (x, r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"], inp["Ws_gu"],
          inp["Ws_down"], valid)
    y_ex, _ = M.experts_forward_mx(*fw, shared_mx=False)
    y_id, _ = M.experts_forward_mx(*fw, shared_mx=False, rnd=adopt)
    args = (x, inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"], inp["Ws_down"], fwd,
            inp["dY"])
    kw = dict(norm_topk=bool(s.norm_topk), aux_coef=s.aux_coef)
    ex = M.backward_mx(*args, **kw)
    idl = M.backward_mx(*args, rnd=adopt, **kw)
    g = lay.grads
    chk = Checker()
    chk.layer("y", lay.bufs["y"], y_ex, y_id)
    names = ["d_logits", "dW_down", "dW_gu", "dx", "dWr"]
    if s.n_shared:
        names += ["dWs_down", "dWs_gu"]
    for n in names:
        chk.layer(n, g[n], ex[n], idl[n])
    adopt.check(chk)
    chk.done()
    if valid is not None:
        pad = inp["valid"] == 0
        assert (g["dx"].cpu()[pad].float() == 0).all()


def test_mx_train_step_differs_from_bf16_layer():
    """The tolerance tells the MX training step from the bf16 layer's: the
    GPU's dx, dW_gu and dW_down are within 1e-2 (Frobenius-relative) of the
    MX oracle with bf16 storage rounding and several times further from the
    bf16 layer's oracle with the same rounding."""
    s = synth.MoEShape("mxtrain", T=600, d=256, E=8, k=2, H=256, n_shared=0, H_shared=0,
                       training=True)
    inp, lay = mx_train_layer(s)
    r, x, valid = route_like_gpu(s, inp, lay)
    fwd = train_fwd(s, inp, r)
    args = (x, inp["Wr"], inp["W_gu"], inp["W_down"], None, None, fwd, inp["dY"])
    mx = M.backward_mx(*args, rnd=bf16_round)
    bf = O.backward(*args, rnd=bf16_round)
    for n in ("dx", "dW_gu", "dW_down"):
        e_mx = frob_err(np64(lay.grads[n]), mx[n])
        e_bf = frob_err(np64(lay.grads[n]), bf[n])
        assert e_mx <= 1e-2 and e_bf > 3 * e_mx, (n, e_mx, e_bf)


def test_mx_train_step_is_deterministic():
    s = scaled_shape(5, 1300, dict(d=512, H=256))
    inp, lay = mx_train_layer(s)
    keep = {n: lay.grads[n].clone() for n in ("dx", "dW_gu", "dW_down", "d_logits")}
    y0 = lay.bufs["y"].clone()
    lay.mx_step(inp["dY"].cuda())
    torch.cuda.synchronize()
    assert torch.equal(y0, lay.bufs["y"])
    for n, v in keep.items():
        assert torch.equal(v, lay.grads[n]), n


@pytest.mark.parametrize("cfg,n_tok", [(5, 3), (2, 8), (4, 3)])
def test_mx_train_full_size_sampled(cfg, n_tok):
    """The training step at its full size, in the calls bench.py times
    (Layer.mx_step): the routing in full, and y, dx and d_logits of a few
    seeded tokens (the last one included) against the MX training oracle
    evaluated on those tokens with the batch's expert loads f; and eight
    columns of dW_down and eight hidden units of dW_gu of one expert, over
    all of that expert's rows."""
    s = synth.shape(cfg)
    inp, lay = mx_train_layer(s)
    b, g = lay.bufs, lay.grads
    x = np64(inp["x"])
    L = O.router_logits(inp["x"], inp["Wr"])
    bias = None if inp["bias"] is None else inp["bias"].numpy().astype(np.float64)
    key = L + (0.0 if bias is None else bias)
    real = np.ones(s.T, bool) if inp["valid"] is None else inp["valid"].numpy() != 0
    sel, _ = reconcile_selection(b["topk_idx"].cpu().numpy(), key,
                                 logit_error_bound(x, np64(inp["Wr"])), s.k, real)
    probs = O.softmax(L)
    r = O.route_stats(probs, sel, real, bool(s.norm_topk))
    np.testing.assert_array_equal(b["topk_idx"].cpu().numpy(), r["topk_idx"])
    offsets, row_offsets, row_of_pair, _ = padded_layout(r["topk_idx"], s.E)
    np.testing.assert_array_equal(b["row_offsets"].cpu().numpy(), row_offsets)
    np.testing.assert_array_equal(b["inv"].cpu().numpy(), row_of_pair)
    chk = Checker()
    # ---- sampled tokens
    rng = np.random.default_rng(100 + cfg)
    ts = np.append(np.sort(rng.choice(s.T - 1, size=n_tok - 1, replace=False)), s.T - 1)
    tsc = torch.from_numpy(ts)
    tsd = tsc.cuda()
    fwd = dict(topk_idx=r["topk_idx"][ts], gates=r["gates"][ts], probs=probs[ts],
               real=real[ts], f=r["f"])
    adopt = AdoptStored(stored_from_layer(lay, True), row_of_pair, s.k, tokens=ts)
    # the forward on the experts the sample chose (renumbered), the backward
    # with the router's own numbering (only chosen experts are quantised)
    topk = fwd["topk_idx"]
    used = np.unique(topk[topk >= 0])
    topk_c = np.where(topk >= 0, np.searchsorted(used, np.maximum(topk, 0)), -1)
    ut = torch.from_numpy(used)
    xs = x[ts]
    ys = {}
    for name, rnd in (("exact", None), ("ideal", adopt)):
        ys[name], _ = M.experts_forward_mx(xs, topk_c, fwd["gates"], inp["W_gu"][ut],
                                           inp["W_down"][ut], inp["Ws_gu"], inp["Ws_down"],
                                           real[ts].astype(np.uint8), shared_mx=False, rnd=rnd)
    chk.layer("y[sample]", b["y"][tsd], ys["exact"], ys["ideal"])
    coef = s.aux_coef * max(int(real[ts].sum()), 1) / int(real.sum())
    args = (xs, inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"], inp["Ws_down"], fwd,
            inp["dY"][tsc])
    ex = M.backward_mx(*args, norm_topk=bool(s.norm_topk), aux_coef=coef)
    idl = M.backward_mx(*args, norm_topk=bool(s.norm_topk), aux_coef=coef, rnd=adopt)
    chk.layer("dx[sample]", g["dx"][tsd], ex["dx"], idl["dx"])
    chk.layer("d_logits[sample]", g["d_logits"][tsd], ex["d_logits"], idl["d_logits"])
    adopt.check(chk)
    # ---- one expert's weight gradients on sampled columns: the MX products
    # restricted to hidden units J (rows of W_gate, W_up and columns of
    # W_down are quantised on their own, and d_out's codes are whole rows, so
    # the restriction is exact)
    e = int(np.argsort(r["counts"])[len(r["counts"]) // 2])
    seg = O.permute(r["topk_idx"], s.E)[1][offsets[e]:offsets[e + 1]]
    tok, slot = seg // s.k, seg % s.k
    gate = r["gates"][tok, slot]
    Wg, Wu = O.split_gu(np64(inp["W_gu"][e]))
    Wd = np64(inp["W_down"][e])
    dY = np64(inp["dY"])
    J = np.sort(rng.choice(s.H, size=8, replace=False))
    xq = M.mx_roundtrip(x[tok])
    qg, qu = M.mx_roundtrip(Wg[J]), M.mx_roundtrip(Wu[J])
    qdk = M.roundtrip_k(Wd[:, J])
    adopt_e = AdoptStored(stored_from_layer(lay, True, cols=J), row_of_pair, s.k)
    res = {}
    for name, rnd in (("exact", None), ("ideal", adopt_e)):
        dWd = np.zeros((s.d, J.size)); dWg = np.zeros((J.size, s.d)); dWu = np.zeros((J.size, s.d))
        for j in range(s.k):
            m = slot == j
            if not m.any():
                continue
            where = dict(e=e, j=j, rows=tok[m])
            a = xq[m] @ qg.T
            bb = xq[m] @ qu.T
            h = O._store(rnd, "h", O.silu(a) * bb, where)
            d_out_v = gate[m][:, None] * dY[tok[m]]
            d_out = O._store(rnd, "d_out", d_out_v, where)
            dH = M._quantised(rnd, "q_d_out", d_out_v, M.mx_roundtrip, where) @ qdk
            da_v, db_v = O.swiglu_backward(dH, M._store16(rnd, "a16", a, where),
                                           M._store16(rnd, "b16", bb, where))
            da, db = O._store(rnd, "da", da_v, where), O._store(rnd, "db", db_v, where)
            dWd += d_out.T @ h
            dWg += da.T @ x[tok[m]]
            dWu += db.T @ x[tok[m]]
        res[name] = (dWd, dWg, dWu)
    jt = torch.from_numpy(J).cuda()
    for nm, gv, k_ in (("dW_down[e]", g["dW_down"][e][:, jt], 0),
                       ("dW_gate[e]", g["dW_gu"][e][jt], 1),
                       ("dW_up[e]", g["dW_gu"][e][jt + s.H], 2)):
        chk.layer(nm, gv, res["exact"][k_], res["ideal"][k_])
    adopt_e.check(chk)
    chk.done()
    del lay
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,shape,bias,valid_real", [
    ("single_token", dict(T=1, d=256, E=8, k=2, H=256, n_shared=1, H_shared=128), None, None),
    ("one_expert_full", dict(T=900, d=256, E=16, k=1, H=256, n_shared=0, H_shared=0),
     [100.0] + [0.0] * 15, None),
    ("half_pad", dict(T=600, d=256, E=8, k=2, H=128, n_shared=1, H_shared=128), None, 300),
])
def test_mx_train_edge_shapes(name, shape, bias, valid_real):
    """The MX training step on one token (one padded 128-row block per
    tensor), on every token sent to one expert (every other expert's
    gradients exactly 0), and on a batch whose second half is PAD (dx and
    d_logits exactly 0 there), against the MX training oracle."""
    s = synth.MoEShape(name, training=True, **shape)
    inp = synth.make_inputs(s, seed=3, with_grad=True)
    if bias is not None:
        inp["bias"] = torch.tensor(bias, dtype=torch.float32)
    if valid_real is not None:
        v = torch.zeros(s.T, dtype=torch.uint8)
        v[:valid_real] = 1
        inp["valid"] = v
    lay = Layer.create(s, training=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    lay.mx_alloc()
    lay.mx_quantize_weights()
    lay.mx_step(dev["dY"])
    torch.cuda.synchronize()
    assert lay.status() == 0
    r, x, valid = route_like_gpu(s, inp, lay)
    np.testing.assert_array_equal(lay.bufs["topk_idx"].cpu().numpy(), r["topk_idx"])
    fwd = train_fwd(s, inp, r)
    adopt = AdoptStored(stored_from_layer(lay, True), padded_layout(r["topk_idx"], s.E)[2], s.k)
    args = (x, inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"], inp["Ws_down"], fwd,
            inp["dY"])
    ex = M.backward_mx(*args, aux_coef=s.aux_coef)
    idl = M.backward_mx(*args, aux_coef=s.aux_coef, rnd=adopt)
    fw = (x, r["topk_idx"], r["gates"], inp["W_gu"], inp["W_down"], inp["Ws_gu"],
          inp["Ws_down"], valid)
    chk = Checker()
    chk.layer("y", lay.bufs["y"], M.experts_forward_mx(*fw, shared_mx=False)[0],
              M.experts_forward_mx(*fw, shared_mx=False, rnd=adopt)[0])
    for n in ("dx", "dW_gu", "dW_down", "d_logits"):
        chk.layer(n, lay.grads[n], ex[n], idl[n])
    adopt.check(chk)
    chk.done()
    g = lay.grads
    if name == "one_expert_full":
        assert not g["dW_gu"][1:].any() and not g["dW_down"][1:].any()
    if valid_real is not None:
        assert not g["dx"][valid_real:].any() and not g["d_logits"][valid_real:].any()


@pytest.mark.parametrize("norm_topk,z_coef", [(0, 0.0), (1, 1e-3)])
def test_mx_train_raw_gates_and_z_loss(norm_topk, z_coef):
    """The MX training step without gate renormalisation, and with the
    router z-loss term, against the MX training oracle (the same router
    terms as the bf16 layer's)."""
    s = synth.scaled(synth.shape(5), T=700, d=512, H=256, norm_topk=norm_topk, z_coef=z_coef)
    inp = synth.make_inputs(s, seed=4, with_grad=True)
    lay = Layer.create(s, training=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    lay.mx_alloc()
    lay.mx_quantize_weights()
    lay.mx_step(dev["dY"])
    torch.cuda.synchronize()
    assert lay.status() == 0
    r, x, valid = route_like_gpu(s, inp, lay)
    np.testing.assert_array_equal(lay.bufs["topk_idx"].cpu().numpy(), r["topk_idx"])
    fwd = train_fwd(s, inp, r)
    fwd["logits"] = O.router_logits(x, inp["Wr"])
    adopt = AdoptStored(stored_from_layer(lay, True), padded_layout(r["topk_idx"], s.E)[2], s.k)
    args = (x, inp["Wr"], inp["W_gu"], inp["W_down"], None, None, fwd, inp["dY"])
    kw = dict(norm_topk=bool(norm_topk), aux_coef=s.aux_coef, z_coef=z_coef)
    ex = M.backward_mx(*args, **kw)
    idl = M.backward_mx(*args, rnd=adopt, **kw)
    chk = Checker()
    for n in ("dx", "dW_gu", "dW_down", "d_logits", "dWr"):
        chk.layer(n, lay.grads[n], ex[n], idl[n])
    adopt.check(chk)
    chk.done()


def test_mx_train_step_needs_no_bf16_ab():
    """The MX training step keeps a | b in its own fp16 buffer (ab16): with
    the bf16 layer's ab left NULL it runs and gives the same gradients bit
    for bit."""
    s = scaled_shape(5, 1300, dict(d=512, H=256))
    inp, lay = mx_train_layer(s)
    keep = {n: lay.grads[n].clone() for n in ("dx", "dW_gu", "dW_down", "d_logits")}
    lay.bufs["ab"] = None
    lay.mx_step(inp["dY"].cuda())
    torch.cuda.synchronize()
    assert lay.status() == 0
    for n, v in keep.items():
        assert torch.equal(v, lay.grads[n]), n
