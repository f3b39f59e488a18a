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
