"""Pins for the MXFP8 oracle (``oracle/mx_oracle.py``): values fixed by the
e4m3 / UE8M0 formats, torch's float8_e4m3fn conversion as a library routine,
brute force, round trips and an independent dense formulation.

A plausible slip (exponent offset 7 instead of 8, ties to odd, no
saturation, blocks along the wrong axis, a dropped h quantisation, the
shared expert left unquantised) fails at least one of them.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import mx_oracle as M


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- e4m3 format

def test_e4m3_table_closed_forms():
    """Values the format fixes: 0x01 is the smallest subnormal 2^-9, 0x07 the
    largest subnormal 7 * 2^-9, 0x08 the smallest normal 2^-6, 0x38 = 1,
    0x7E = 448 the largest finite; strictly increasing."""
    t = M.e4m3_table()
    assert t.shape == (127,)
    assert t[0] == 0.0 and t[1] == 2.0 ** -9 and t[7] == 7 * 2.0 ** -9
    assert t[8] == 2.0 ** -6 and t[0x38] == 1.0 and t[0x7E] == 448.0
    assert (np.diff(t) > 0).all()


def test_e4m3_decode_matches_torch_float8():
    """Decoding every code agrees with torch.float8_e4m3fn (a library
    routine), NaN codes included."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = M.e4m3_decode(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_e4m3_round_matches_torch_float8():
    """Rounding within the finite range agrees with torch's round-to-nearest-
    even conversion to float8_e4m3fn: random values, every midpoint between
    neighbouring codes (the ties), and the codes themselves."""
    t = M.e4m3_table()
    mids = (t[1:] + t[:-1]) / 2
    rng = _rng(0)
    v = np.concatenate([t, mids, -mids, rng.uniform(-448, 448, 20000),
                        rng.standard_normal(20000) * 2.0 ** rng.integers(-12, 8, 20000)])
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(M.e4m3_round(v), ref)


def test_e4m3_round_saturates_and_keeps_sign():
    assert M.e4m3_round(np.array([500.0, 1e9, -470.0])).tolist() == [0x7E, 0x7E, 0xFE]
    assert M.e4m3_round(np.array([0.0, -0.0, -1e-6])).tolist() == [0x00, 0x80, 0x80]


# ---------------------------------------------------------------- MX blocks

def test_mx_scale_closed_forms():
    """X = floor(log2 amax) - 8: amax 1 -> X -8 (byte 119, element 256 ->
    code 0x78); amax 448 -> X 0 (448 itself, 0x7E); amax 500 -> X 0 and the
    500 saturates to 448; amax just below 2 -> X -8; zero block -> byte 0."""
    def q(block):
        c, s = M.mx_quantize(np.asarray(block, dtype=np.float64)[None, :])
        return c[0], int(s[0, 0])

    c, s = q(np.ones(32))
    assert s == 119 and (c == 0x78).all()          # 1 / 2^-8 = 256 = 1.0 * 2^8
    c, s = q([448.0] + [0.0] * 31)
    assert s == 127 and c[0] == 0x7E and (c[1:] == 0).all()
    c, s = q([500.0] + [1.0] * 31)
    assert s == 127 and c[0] == 0x7E and (c[1:] == 0x38).all()
    c, s = q([1.9921875] + [0.0] * 31)             # bf16 value just below 2
    assert s == 119
    c, s = q(np.zeros(32))
    assert s == 0 and (c == 0).all()


def test_mx_quantize_is_nearest_on_the_block_grid():
    """Brute force: each element's dequantised value is the nearest of all
    253 finite values code * 2^X of its block (ties to the even code), or
    +-448 * 2^X where it lies beyond; X follows the closed form."""
    rng = _rng(1)
    grid_mag = M.e4m3_table()
    for trial in range(40):
        scale = 2.0 ** rng.integers(-20, 20)
        v = rng.standard_normal(32) * scale
        if trial % 4 == 0:
            v[rng.integers(32)] = 0.0
        c, s = M.mx_quantize(v[None, :])
        X = int(s[0, 0]) - 127
        amax = np.abs(v).max()
        assert 2.0 ** (X + 8) <= amax < 2.0 ** (X + 9)
        deq = M.mx_dequantize(c, s)[0]
        for i in range(32):
            a = min(abs(v[i]) / 2.0 ** X, 448.0)
            dist = np.abs(grid_mag - a)
            best = np.flatnonzero(dist == dist.min())
            pick = best[0] if best.size == 1 else [b for b in best if b % 2 == 0][0]
            assert abs(deq[i]) == grid_mag[pick] * 2.0 ** X
            assert np.signbit(deq[i]) == np.signbit(v[i])


def test_mx_representable_blocks_round_trip():
    """A block made of e4m3 values times 2^X, with its largest magnitude in
    [256, 448], quantises back to the same codes and the same scale."""
    rng = _rng(2)
    for _ in range(50):
        X = int(rng.integers(-30, 30))
        codes = rng.integers(0, 256, 32).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x10
        codes[rng.integers(32)] = 0x78 | int(rng.integers(0, 7))   # magnitude 256..448
        v = M.e4m3_decode(codes) * 2.0 ** X
        c, s = M.mx_quantize(v[None, :])
        assert int(s[0, 0]) == X + 127
        np.testing.assert_array_equal(np.abs(M.e4m3_decode(c[0])), np.abs(M.e4m3_decode(codes)))


def test_mx_blocks_are_rows_of_32():
    """Blocks run along the last axis, 32 at a time: changing one block of
    one row changes only that block's codes and scale."""
    rng = _rng(3)
    v = rng.standard_normal((64, 128))
    c0, s0 = M.mx_quantize(v)
    assert c0.shape == (64, 128) and s0.shape == (64, 4)
    w = v.copy()
    w[2, 32:64] *= 1000.0
    c1, s1 = M.mx_quantize(w)
    assert s1.shape == (64, 4)
    changed = np.argwhere((c0 != c1).reshape(64, 4, 32).any(-1) | (s0 != s1))
    assert changed.tolist() == [[2, 1]]


# ---------------------------------------------------------------- MX experts

def _tiny(seed, T=24, d=64, E=4, k=2, H=64, shared=True):
    rng = _rng(seed)
    x = rng.standard_normal((T, d))
    W_gu = rng.standard_normal((E, 2 * H, d)) * 0.2
    W_down = rng.standard_normal((E, d, H)) * 0.2
    Ws_gu = rng.standard_normal((2 * H, d)) * 0.2 if shared else None
    Ws_down = rng.standard_normal((d, H)) * 0.2 if shared else None
    logits = rng.standard_normal((T, E)).astype(np.float32)
    r = O.route(logits, k)
    return x, W_gu, W_down, Ws_gu, Ws_down, r


def test_mx_experts_dense_masked_formulation():
    """Independent formulation: every expert applied to every token on the
    quantised operands, y_t = sum_e [e selected] g_{t,e} F^mx_e(x_t) + the
    shared FFN on quantised operands, written out with explicit quantise
    steps."""
    x, W_gu, W_down, Ws_gu, Ws_down, r = _tiny(4)
    y, _ = M.experts_forward_mx(x, r["topk_idx"], r["gates"], W_gu, W_down, Ws_gu, Ws_down)
    T, d = x.shape
    E, H2, _ = W_gu.shape
    H = H2 // 2
    xc, xs = M.mx_quantize(x)
    xq = M.mx_dequantize(xc, xs)
    ref = np.zeros((T, d))
    for e in range(E):
        gc, gs = M.mx_quantize(W_gu[e])
        Wq = M.mx_dequantize(gc, gs)
        dc, ds = M.mx_quantize(W_down[e])
        Wdq = M.mx_dequantize(dc, ds)
        a = xq @ Wq[:H].T
        b = xq @ Wq[H:].T
        h = a / (1.0 + np.exp(-a)) * b
        hq = M.mx_dequantize(*M.mx_quantize(h))
        out = hq @ Wdq.T
        w = ((r["topk_idx"] == e) * r["gates"]).sum(axis=1)
        ref += w[:, None] * out
    sc, ss = M.mx_quantize(Ws_gu)
    Wsq = M.mx_dequantize(sc, ss)
    a = xq @ Wsq[:H].T
    b = xq @ Wsq[H:].T
    hs = M.mx_dequantize(*M.mx_quantize(a / (1.0 + np.exp(-a)) * b))
    ref += hs @ M.mx_dequantize(*M.mx_quantize(Ws_down)).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_mx_experts_close_to_exact_and_not_equal():
    """MX quantisation moves the routed and the shared outputs by a few
    percent of their scale (3 mantissa bits: at most 1/16 relative per
    element), never by more, and does move them."""
    x, W_gu, W_down, Ws_gu, Ws_down, r = _tiny(5)
    y_mx, routed_mx = M.experts_forward_mx(x, r["topk_idx"], r["gates"], W_gu, W_down)
    y, routed = O.experts_forward(x, r["topk_idx"], r["gates"], W_gu, W_down)
    rel = np.abs(routed_mx - routed).max() / np.abs(routed).max()
    assert 1e-3 < rel < 0.2
    ys_mx, _ = M.experts_forward_mx(x, r["topk_idx"], r["gates"], W_gu, W_down, Ws_gu, Ws_down)
    ys, _ = O.experts_forward(x, r["topk_idx"], r["gates"], W_gu, W_down, Ws_gu, Ws_down)
    shared_mx, shared = ys_mx - y_mx, ys - y
    rel = np.abs(shared_mx - shared).max() / np.abs(shared).max()
    assert 1e-3 < rel < 0.2


def test_mx_experts_exact_on_representable_operands():
    """With x and the weights already MX-representable and h quantised
    exactly (a = 0 gives h = 0), the MX forward equals the exact forward."""
    x, W_gu, W_down, _, _, r = _tiny(6, shared=False)
    xq = M.mx_roundtrip(x)
    Wq = M.mx_roundtrip(W_gu)
    Wq[:, : Wq.shape[1] // 2] = 0.0                 # gate rows 0 -> h = 0
    Wdq = M.mx_roundtrip(W_down)
    y_mx, _ = M.experts_forward_mx(xq, r["topk_idx"], r["gates"], Wq, Wdq)
    y, _ = O.experts_forward(xq, r["topk_idx"], r["gates"], Wq, Wdq)
    np.testing.assert_array_equal(y_mx, y)
    assert (y == 0).all()


def test_mx_rejects_ragged_blocks():
    with pytest.raises(ValueError):
        M.mx_quantize(np.ones((2, 48)))


# ------------------------------------------------ MX training step (backward)

def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(
        torch.bfloat16).double().numpy()


def _train_case(seed, T=20, d=64, E=4, k=2, H=96, shared=True, norm=True):
    """A tiny layer whose sizes are all different (d, H, 2H, rows), so a
    quantised operand's last axis tells which product it serves."""
    rng = _rng(seed)
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((d, E)) * 0.3
    W_gu = rng.standard_normal((E, 2 * H, d)) * 0.2
    W_down = rng.standard_normal((E, d, H)) * 0.2
    Ws_gu = rng.standard_normal((2 * H, d)) * 0.2 if shared else None
    Ws_down = rng.standard_normal((d, H)) * 0.2 if shared else None
    dY = rng.standard_normal((T, d))
    fwd = M.forward_mx_train(x, Wr, W_gu, W_down, Ws_gu, Ws_down, k=k, norm_topk=norm)
    return x, Wr, W_gu, W_down, Ws_gu, Ws_down, dY, fwd


@pytest.mark.parametrize("norm", [True, False])
def test_mx_backward_is_the_bf16_backward_with_bf16_rounding(norm):
    """With the MX round trip replaced by a bf16 round trip and inputs that
    bf16 holds exactly, the MX training step's backward is the bf16 layer's
    backward (pinned by finite differences and the storage pins), term for
    term, once the bf16 layer's routed experts also keep a and b in fp16 (as
    the MX step does) instead of bf16: Q(h) in the down
    product plays the bf16 layer's stored h, Q(d_out) and Q(d_gu) its stored
    d_out and d_gu, and the other quantised operands are bf16 values
    already."""
    x, Wr, W_gu, W_down, Ws_gu, Ws_down, dY, fwd = _train_case(7, norm=norm)
    x, W_gu, W_down, Ws_gu, Ws_down, dY = map(_bf16, (x, W_gu, W_down, Ws_gu, Ws_down, dY))
    fwd = M.forward_mx_train(x, Wr, W_gu, W_down, Ws_gu, Ws_down, k=2, norm_topk=norm)
    args = (x, Wr, W_gu, W_down, Ws_gu, Ws_down, fwd, dY)
    got = M.backward_mx(*args, norm_topk=norm, rnd=_bf16, quant=_bf16)

    class RoutedABInFp16:
        def store(self, point, v, where):
            if point in ("a", "b") and not where.get("shared"):
                return M.fp16_round(v)
            return _bf16(v)
    ref = O.backward(*args, norm_topk=norm, rnd=RoutedABInFp16())
    for n in ("dx", "dWr", "dW_gu", "dW_down", "dWs_gu", "dWs_down", "d_logits", "dg"):
        np.testing.assert_allclose(got[n], ref[n], rtol=1e-12, atol=1e-12, err_msg=n)


def test_mx_training_forward_has_the_bf16_shared_expert():
    """The training step's forward: the routed experts' MX sum plus the bf16
    layer's shared expert (its hidden through the storage hook)."""
    x, Wr, W_gu, W_down, Ws_gu, Ws_down, dY, fwd = _train_case(11)
    y_t, _ = M.experts_forward_mx(x, fwd["topk_idx"], fwd["gates"], W_gu, W_down, Ws_gu,
                                  Ws_down, shared_mx=False, rnd=_bf16)
    y_r, _ = M.experts_forward_mx(x, fwd["topk_idx"], fwd["gates"], W_gu, W_down, rnd=_bf16)
    sg, su = O.split_gu(Ws_gu)
    shared, *_ = O.swiglu_parts(x, sg, su, Ws_down, _bf16)
    np.testing.assert_allclose(y_t - y_r, shared, rtol=1e-12, atol=1e-12)


class _AxisSpy:
    """A quantiser that records the shape of every array it quantises (its
    last axis is the one quantised) and then quantises it."""

    def __init__(self):
        self.shapes = []

    def __call__(self, v):
        v = np.asarray(v, dtype=np.float64)
        self.shapes.append(v.shape)
        return M.mx_roundtrip(v)


def test_mx_backward_quantises_each_operand_along_its_reduction_axis():
    """Every product of a routed expert's MX step quantises its operands in
    blocks along the axis it sums over: the forward a, b over d (x rows and
    W_gate, W_up rows: last axis d), out over H (h rows, W_down rows: last
    axis H); the data gradients dH over d (d_out rows [n][d] and W_down^T
    [H][d]) and dx over 2H (d_gu rows [n][2H] and W_gu^T [d][2H]).  With
    d = 64, H = 96, 2H = 192 and groups of other sizes, the shapes show it."""
    x, Wr, W_gu, W_down, Ws_gu, Ws_down, dY, fwd = _train_case(8, shared=False)
    d, H = 64, 96
    spy = _AxisSpy()
    M.backward_mx(x, Wr, W_gu, W_down, None, None, fwd, dY, rnd=_bf16, quant=spy)
    assert spy.shapes[0] == x.shape                           # Q(x), once
    rest = spy.shapes[1:]
    # per expert with rows: its weights once -- W_gate, W_up [H][d], W_down
    # [d][H], W_down^T [H][d], W_gu^T [d][2H] -- then per group of n rows
    # h [n][H], d_out [n][d], d_gu [n][2H]
    weights = [(H, d), (H, d), (d, H), (H, d), (d, 2 * H)]
    i = n_experts = n_groups = 0
    while i < len(rest):
        assert rest[i:i + 5] == weights, rest[i:i + 5]
        i += 5
        n_experts += 1
        while i < len(rest) and rest[i:i + 5] != weights:
            n = rest[i][0]
            assert rest[i:i + 3] == [(n, H), (n, d), (n, 2 * H)], rest[i:i + 3]
            i += 3
            n_groups += 1
    idx = fwd["topk_idx"]
    assert n_experts == len(np.unique(idx[idx >= 0]))
    assert n_groups == sum(len(np.unique(idx[:, j][idx[:, j] >= 0])) for j in range(idx.shape[1]))


def test_mx_backward_dense_masked_formulation():
    """Independent formulation of the routed data gradients: every expert on
    every token, masked by the selection, with each quantise step written
    out: dx_t = sum_e [e selected at slot j] Q(swiglu_bwd(Q(g dY_t)
    Q_d(W_down_e), fp16 a, fp16 b)) Q_2H(W_gu_e), plus the shared expert and
    the router terms of the bf16 layer.  The MX operands are quantised from
    the unrounded d_out and d_gu (only the weight gradients take bf16
    copies), and the chain rule takes a and b in fp16."""
    x, Wr, W_gu, W_down, Ws_gu, Ws_down, dY, fwd = _train_case(9, shared=False)
    got = M.backward_mx(x, Wr, W_gu, W_down, None, None, fwd, dY, rnd=_bf16)
    T, d = x.shape
    E, H2, _ = W_gu.shape
    H = H2 // 2
    Q = M.mx_roundtrip
    xq = Q(x)
    dx = np.zeros((T, d))
    dg = np.zeros(fwd["topk_idx"].shape)
    for e in range(E):
        Wg, Wu = W_gu[e][:H], W_gu[e][H:]
        a = xq @ Q(Wg).T
        b = xq @ Q(Wu).T
        out = _bf16(Q(a / (1 + np.exp(-a)) * b) @ Q(W_down[e]).T)   # kept in bf16
        WdT = Q(W_down[e].T)                 # rows of W_down^T: blocks along d
        WguT = Q(W_gu[e].T)                  # rows of W_gu^T: blocks along 2H
        for j in range(fwd["topk_idx"].shape[1]):
            m = fwd["topk_idx"][:, j] == e
            gte = np.where(m, fwd["gates"][:, j], 0.0)
            dg[:, j] += np.where(m, (dY * out).sum(axis=1), 0.0)
            dH = Q(gte[:, None] * dY) @ WdT.T       # d_out quantised from g dY itself
            a16, b16 = M.fp16_round(a), M.fp16_round(b)
            sa = 1 / (1 + np.exp(-a16))
            da = dH * b16 * sa * (1 + a16 * (1 - sa))
            db = dH * a16 * sa
            dx += np.where(m[:, None], _bf16(Q(np.concatenate([da, db], axis=1)) @ WguT.T), 0.0)
    dL = O.router_logit_grad(dg, fwd["topk_idx"], fwd["gates"], fwd["probs"], True)
    dL += O.aux_logit_grad(fwd["probs"], fwd["f"], fwd["real"], 0.01)
    dx += dL @ Wr.T
    np.testing.assert_allclose(got["dg"], dg, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got["dx"], dx, rtol=1e-11, atol=1e-11)


def test_mx_backward_differs_from_bf16_by_the_quantisation():
    """The MX data gradients move dx by a few percent of its scale against
    the bf16 layer's, never more, and do move it; the weight gradients of
    the bf16 wgrad products move only through their MX-forward inputs."""
    x, Wr, W_gu, W_down, Ws_gu, Ws_down, dY, fwd = _train_case(10)
    args = (x, Wr, W_gu, W_down, Ws_gu, Ws_down, fwd, dY)
    mx = M.backward_mx(*args, rnd=_bf16)
    bf = O.backward(*args, rnd=_bf16)
    rel = np.abs(mx["dx"] - bf["dx"]).max() / np.abs(bf["dx"]).max()
    assert 1e-3 < rel < 0.2
    np.testing.assert_allclose(mx["dWs_gu"], bf["dWs_gu"], rtol=1e-12, atol=1e-12)


class _QuantSpy:
    """Storage hook (bf16) with the quantisation-point method: records each
    point with its shape and group, checks that the oracle hands it Q(v),
    and returns Q(v) or, for the points in ``override``, override(Q(v))."""

    def __init__(self, override=None):
        self.seen = []
        self.override = override or {}

    def __call__(self, v):
        return _bf16(v)

    def quantised(self, point, v, q, where):
        self.seen.append((point, v.shape, where["e"], where["j"]))
        np.testing.assert_array_equal(q, M.mx_roundtrip(v))
        return self.override.get(point, lambda a: a)(q)


def test_mx_quantisation_points_feed_their_products():
    """The hook sees Q(h), Q(d_out) and Q(d_gu) once per (expert, slot)
    group, in that order and with the group's rows, and what it returns is
    what the products use: Q(d_gu) only the routed dx, Q(d_out) the dH
    product (so da, db and dW_gu) but not dW_down, and Q(h) only dg."""
    x, Wr, W_gu, W_down, Ws_gu, Ws_down, dY, fwd = _train_case(8, shared=False)
    d, H = 64, 96
    args = (x, Wr, W_gu, W_down, None, None, fwd, dY)
    spy = _QuantSpy()
    base = M.backward_mx(*args, rnd=spy)
    pts = [p for p, *_ in spy.seen]
    assert pts == ["q_h", "q_d_out", "q_d_gu"] * (len(pts) // 3) and pts
    for i in range(0, len(spy.seen), 3):
        (_, sh, e, j), (_, sd, e2, j2), (_, sg, e3, j3) = spy.seen[i:i + 3]
        n = int((fwd["topk_idx"][:, j] == e).sum())
        assert (sh, sd, sg) == ((n, H), (n, d), (n, 2 * H)) and (e, j) == (e2, j2) == (e3, j3)
    router_dx = base["d_logits"] @ np.asarray(Wr, dtype=np.float64).T
    z = M.backward_mx(*args, rnd=_QuantSpy({"q_d_gu": np.zeros_like}))
    np.testing.assert_allclose(z["dx"], router_dx, rtol=1e-12, atol=1e-12)
    for n in ("dW_gu", "dW_down", "d_logits"):
        np.testing.assert_array_equal(z[n], base[n])
    z = M.backward_mx(*args, rnd=_QuantSpy({"q_d_out": np.zeros_like}))
    assert not z["dW_gu"].any()
    np.testing.assert_allclose(z["dx"], router_dx, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(z["dW_down"], base["dW_down"])
    z = M.backward_mx(*args, rnd=_QuantSpy({"q_h": np.zeros_like}))
    assert not z["dg"].any()
    for n in ("dW_gu", "dW_down"):
        np.testing.assert_array_equal(z[n], base[n])
    # the forward: Q(h) per group, and a zero Q(h) leaves no routed output
    spy = _QuantSpy()
    y0, _ = M.experts_forward_mx(x, fwd["topk_idx"], fwd["gates"], W_gu, W_down, rnd=spy)
    assert [p for p, *_ in spy.seen] == ["q_h"] * len(spy.seen) and spy.seen
    y1, _ = M.experts_forward_mx(x, fwd["topk_idx"], fwd["gates"], W_gu, W_down,
                                 rnd=_QuantSpy({"q_h": np.zeros_like}))
    assert y0.any() and not y1.any()


def test_fp16_round_by_hand():
    """The binary16 rounding of the chain rule's a and b: ties to even at 1
    (ulp 2^-10), the binade edge, subnormals (spacing 2^-24), a value of
    ulp 1/2, and the clamp at the largest finite value."""
    r = M.fp16_round
    assert r(1 + 2.0 ** -11) == 1.0                       # tie -> even (1.0)
    assert r(1 + 3 * 2.0 ** -11) == 1 + 2.0 ** -9         # tie -> even mantissa
    assert r(1 + 2.0 ** -11 + 2.0 ** -30) == 1 + 2.0 ** -10
    assert r(-(2 - 2.0 ** -12)) == -2.0                   # rounds up into the next binade
    assert r(2.0 ** -24) == 2.0 ** -24 and r(2.0 ** -26) == 0.0
    assert r(3 * 2.0 ** -26) == 2.0 ** -24                # 0.75 of the smallest subnormal
    assert r(1000.3) == 1000.5 and r(1000.2) == 1000.0    # spacing 1/2 in [512, 1024)
    assert r(65504.0) == 65504.0 and r(7e4) == 65504.0 and r(-1e9) == -65504.0
