"""CPU fp64 oracle of the MXFP8 expert forward.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
of ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import or
run this module.  It shares no code with the CUDA path and never imports it.

What it follows:

* "KohakUwULLM" README, Key features: native MXFP8 training with e4m3 values
  and UE8M0 scales, one scale per block of 32 consecutive values, applied to
  the feed-forward pair and the routed experts, with fully fused MXFP8 expert
  kernels.
* The element and scale formats themselves (the pages name them only): e4m3
  is the 8-bit float with 1 sign bit, 4 exponent bits of bias 7 and 3
  mantissa bits, subnormals at exponent field 0, no infinities and NaN at
  S.1111.111, so the largest finite magnitude is 1.75 * 2^8 = 448.  UE8M0 is
  an 8-bit biased exponent (bias 127, 0xFF reserved): the scale 2^(byte-127).

Readings (the pages say only "e4m3 values with UE8M0 per-32 block scales"):

* Blocks run along the reduction axis of each product: x rows and W_gu rows
  along d, the hidden h rows and W_down rows along H.
* A block's shared exponent is X = floor(log2(max |v|)) - 8 (8 being the
  exponent of the largest e4m3 normal), clamped to [-127, 127]; an all-zero
  block takes X = -127.  Each element is v / 2^X rounded to the nearest e4m3
  value, ties to the even code, and magnitudes above 448 saturate to 448.
* The routed experts and the shared expert (the layer's dense feed-forward
  pair) run on MXFP8 operands: a = Q(x) Q(W_gate)^T, b = Q(x) Q(W_up)^T,
  h = silu(a) * b, out = Q(h) Q(W_down)^T, with Q the quantise-dequantise
  round trip above and everything else exact (fp64).  The router and the
  combine are unchanged (no MX).

Pins: ``tests/test_oracle_mx.py`` (closed forms, torch's float8_e4m3fn
conversion as a library routine, brute-force nearest rounding, round trips of
representable blocks, row independence, and the dense-masked formulation of
the MX expert sum).
"""
from __future__ import annotations

import numpy as np

from . import moe_oracle as mo

f64 = np.float64
E4M3_MAX = 448.0
BLOCK = 32


def e4m3_table():
    """Magnitudes of the 127 non-negative finite e4m3 codes 0x00..0x7E, in
    code order (which is increasing value order)."""
    c = np.arange(127)
    e = c >> 3
    m = c & 7
    return np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))


def e4m3_decode(codes):
    """uint8 e4m3 codes -> float64 (NaN for the NaN codes)."""
    c = np.asarray(codes).astype(np.int64)
    mag = c & 0x7F
    tab = np.append(e4m3_table(), np.nan)
    v = tab[mag]
    return np.where(c & 0x80, -v, v)


def e4m3_round(q):
    """Round float64 values to e4m3 codes: nearest value, ties to the even
    code, magnitudes above 448 saturate to 448; the sign bit is q's."""
    q = np.asarray(q, dtype=f64)
    tab = e4m3_table()
    a = np.minimum(np.abs(q), E4M3_MAX)
    i = np.clip(np.searchsorted(tab, a, side="left"), 1, 126)  # tab[i-1] < a <= tab[i]
    lo, hi = tab[i - 1], tab[i]
    d_lo, d_hi = a - lo, hi - a
    up = (d_hi < d_lo) | ((d_hi == d_lo) & (i % 2 == 0))
    code = np.where(up, i, i - 1)
    return (code | (np.signbit(q).astype(np.int64) << 7)).astype(np.uint8)


def mx_scale_exp(amax):
    """Shared block exponent X = floor(log2 amax) - 8, clamped to [-127, 127];
    -127 for amax = 0.  frexp gives floor(log2) exactly."""
    amax = np.asarray(amax, dtype=f64)
    _, e = np.frexp(amax)                    # amax = m 2^e, m in [0.5, 1)
    X = np.where(amax > 0, e - 1 - 8, -127)
    return np.clip(X, -127, 127).astype(np.int64)


def mx_quantize(v):
    """Blocks of 32 along the last axis (length a multiple of 32) ->
    (codes uint8, same shape as v; scale bytes uint8, [..., K/32])."""
    v = np.asarray(v, dtype=f64)
    K = v.shape[-1]
    if K % BLOCK:
        raise ValueError("the quantised axis must be a multiple of 32")
    b = v.reshape(v.shape[:-1] + (K // BLOCK, BLOCK))
    X = mx_scale_exp(np.abs(b).max(axis=-1))
    q = b / np.exp2(X.astype(f64))[..., None]     # exact: a power-of-two scaling
    return e4m3_round(q).reshape(v.shape), (X + 127).astype(np.uint8)


def mx_dequantize(codes, scales):
    """Inverse of :func:`mx_quantize` on its own outputs: value * 2^(byte-127)."""
    v = e4m3_decode(codes)
    K = v.shape[-1]
    b = v.reshape(v.shape[:-1] + (K // BLOCK, BLOCK))
    s = np.exp2(np.asarray(scales).astype(f64) - 127.0)
    return (b * s[..., None]).reshape(v.shape)


def mx_roundtrip(v):
    """Q(v): quantise to MXFP8 along the last axis and back to float64."""
    return mx_dequantize(*mx_quantize(v))


def experts_forward_mx(x, topk_idx, gates, W_gu, W_down, Ws_gu=None, Ws_down=None,
                       valid=None):
    """The expert sum of the layer with MXFP8 experts.

    Routed part: the permute/combine formulation of ``moe_oracle`` on the
    quantised operands Q(x), Q(W_gu) (blocks along d) and Q(W_down) (blocks
    along H), with the hidden h quantised along H before the down product.
    The shared expert is the same SwiGLU on Q(x), Q(Ws_gu), Q(Ws_down) with
    its hidden quantised along its width, on real tokens.
    Returns (y [T][d], routed [T][k][d])."""
    x = mo._f64(x)
    xq = mx_roundtrip(x)
    y, routed = mo.experts_forward(xq, topk_idx, gates, mx_roundtrip(mo._f64(W_gu)),
                                   mx_roundtrip(mo._f64(W_down)), valid=valid,
                                   rnd=mx_roundtrip)
    if Ws_gu is not None:
        real = np.ones(x.shape[0], dtype=bool) if valid is None else (
            np.asarray(mo._np(valid)) != 0)
        sg, su = mo.split_gu(mx_roundtrip(mo._f64(Ws_gu)))
        shared, *_ = mo.swiglu_parts(xq[real], sg, su, mx_roundtrip(mo._f64(Ws_down)),
                                     rnd=mx_roundtrip)
        y[real] += shared
    return y, routed


def forward_mx(x, Wr, W_gu, W_down, Ws_gu=None, Ws_down=None, k=2, bias=None,
               valid=None, norm_topk=True, logits=None):
    """Whole layer with MXFP8 experts: the router and route of
    ``moe_oracle.forward`` (fp32 logits, unchanged), then the MX expert sum."""
    if logits is None:
        logits = mo.router_logits(x, Wr).astype(np.float32)
    r = mo.route(logits, k, bias=bias, valid=valid, norm_topk=norm_topk)
    y, routed = experts_forward_mx(x, r["topk_idx"], r["gates"], W_gu, W_down, Ws_gu,
                                   Ws_down, valid)
    r.update(y=y, routed=routed, logits=np.asarray(logits))
    return r
