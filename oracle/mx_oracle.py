"""CPU fp64 oracle of the MXFP8 experts: the forward, and the training
step whose routed experts run in MXFP8 (:func:`backward_mx`).

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
* The training step (:func:`backward_mx`, "KohakUwULLM" README, Key features
  and Selected measurements: MXFP8 training of the MoE experts) puts the
  routed experts' two data-gradient products on MXFP8 operands, each one
  rounding of its own value, and keeps the weight gradients, the shared
  expert and the router in the bf16 layer's form; its docstring states the
  reading in full.

Pins: ``tests/test_oracle_mx.py`` (closed forms, torch's float8_e4m3fn
conversion as a library routine, brute-force nearest rounding, round trips of
representable blocks, row independence, the dense-masked formulation of the
MX expert sum; for the training step the reduction to the bf16 layer's
backward when the round trip is a bf16 one, the axis of every quantised
operand, a dense-masked formulation of the MX data gradients, the
quantisation points of the storage hook, and binary16 rounding by hand).
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
                       valid=None, shared_mx=True, rnd=None):
    """The expert sum of the layer with MXFP8 experts.

    Routed part: the permute/combine formulation of ``moe_oracle`` on the
    quantised operands Q(x), Q(W_gu) (blocks along d) and Q(W_down) (blocks
    along H), with the hidden h quantised along H before the down product.
    The shared expert is the same SwiGLU on Q(x), Q(Ws_gu), Q(Ws_down) with
    its hidden quantised along its width, on real tokens; with shared_mx
    False it is the bf16 layer's (exact operands, its hidden through the
    storage hook ``rnd``), as in the MXFP8 training step (:func:`backward_mx`).
    Returns (y [T][d], routed [T][k][d])."""
    x = mo._f64(x)
    xq = mx_roundtrip(x)
    y, routed = mo.experts_forward(xq, topk_idx, gates, mx_roundtrip(mo._f64(W_gu)),
                                   mx_roundtrip(mo._f64(W_down)), valid=valid,
                                   rnd=_HiddenMX(rnd))
    if Ws_gu is not None:
        real = np.ones(x.shape[0], dtype=bool) if valid is None else (
            np.asarray(mo._np(valid)) != 0)
        if shared_mx:
            sg, su = mo.split_gu(mx_roundtrip(mo._f64(Ws_gu)))
            shared, *_ = mo.swiglu_parts(xq[real], sg, su, mx_roundtrip(mo._f64(Ws_down)),
                                         rnd=mx_roundtrip)
        else:
            sg, su = mo.split_gu(mo._f64(Ws_gu))
            rows = np.nonzero(real)[0]
            shared, *_ = mo.swiglu_parts(x[real], sg, su, mo._f64(Ws_down), rnd,
                                         dict(shared=True, rows=rows))
        y[real] += shared
    return y, routed


class _HiddenMX:
    """The routed hidden's MX rounding in the form of ``moe_oracle``'s
    storage hook: Q(h) at the quantisation point "q_h" (:func:`_quantised`,
    so that the hook ``rnd`` may see it)."""

    def __init__(self, rnd):
        self.rnd = rnd

    def store(self, point, v, where):
        if point != "h":                      # the other storage points: the hook's
            return mo._store(self.rnd, point, v, where)
        return _quantised(self.rnd, "q_h", v, mx_roundtrip, where)


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


# --------------------------------------------------------------------------
# Training step with MXFP8 routed experts
# --------------------------------------------------------------------------

def fp16_round(v):
    """v rounded to IEEE binary16 (11 significant bits, round to nearest
    even, subnormals below 2^-14) and back to float64; magnitudes past the
    largest finite binary16, 65504, are clamped to it."""
    v = np.clip(np.asarray(v, dtype=f64), -65504.0, 65504.0)
    return v.astype(np.float16).astype(f64)


def _store16(rnd, point, v, where):
    """a or b as the MXFP8 training step keeps them for the chain rule, at
    storage point ``point`` ("a16", "b16"): with the storage hook's store()
    form the hook sees the point; a plain rounding callable means storage
    rounding is on, and these points round to binary16 (:func:`fp16_round`);
    None keeps v.  No arithmetic happens here."""
    if rnd is None:
        return v
    if hasattr(rnd, "store"):
        return rnd.store(point, v, where)
    return fp16_round(v)


def _quantised(rnd, point, v, quant, where):
    """Q(v) at a quantisation point of a routed expert ("q_h", "q_d_out" or
    "q_d_gu", rows ``where``): ``quant(v)``, or ``rnd.quantised(point, v,
    quant(v), where)`` when the storage hook has that method.  No arithmetic
    happens here."""
    q = quant(v)
    if rnd is not None and hasattr(rnd, "quantised"):
        return rnd.quantised(point, v, q, where)
    return q


def roundtrip_k(W, quant=None):
    """Q along axis 0 of a [K][N] matrix: the operand of ``v @ W`` quantised
    in blocks of 32 along the product's reduction axis K."""
    quant = quant or mx_roundtrip
    return quant(np.asarray(W, dtype=f64).T).T


def backward_mx(x, Wr, W_gu, W_down, Ws_gu, Ws_down, fwd, dY, norm_topk=True,
                aux_coef=0.01, rnd=None, z_coef=0.0, quant=None):
    """Gradients of J = <dY, y> + aux_coef * aux + z_coef * z_loss for the
    layer whose routed experts run in MXFP8, by the chain rule.

    Readings (the pages name MXFP8 training of the routed experts and the
    formats only):

    * Forward of a routed expert: a = Q(x) Q(W_gate)^T, b = Q(x) Q(W_up)^T,
      h = silu(a) b, out = Q(h) Q(W_down)^T (as :func:`experts_forward_mx`).
    * The data-gradient products run on MXFP8 operands quantised in blocks of
      32 along each product's reduction axis: dH = Q(d_out) Qk(W_down) with
      d_out = g dY (reduction over d), and dx = Q(d_gu) Qk(W_gu) with
      d_gu = [da | db] (reduction over 2H); Qk quantises a weight along the
      axis the product sums over (:func:`roundtrip_k`).
    * Q(d_out) and Q(d_gu) quantise the values themselves, once: d_out = g dY
      and the chain rule's [da | db] as computed, not their bf16 copies (a
      bf16 rounding before the e4m3 one would move about 2% of the codes by
      a whole e4m3 step).  For the same reason the chain rule takes a and b
      at fp16 storage points ("a16", "b16": 11 significant bits to bf16's 8,
      which makes such moves about 8 times rarer).
    * The weight-gradient products take the saved h, d_out, d_gu and x at
      the bf16 storage points of the bf16 layer (``rnd``, the hook of
      ``moe_oracle.backward``; h here is the hidden before its MX rounding),
      and each slot's expert output and dx contribution are kept in bf16
      before the slots are summed, as there ("out", "dxe").
    * The quantisations of h, d_out and d_gu are points of the same hook
      (:func:`_quantised`: "q_h", "q_d_out", "q_d_gu"), so that a test can
      continue from another valid quantisation.
    * The shared expert, the router and the routing gradient are the bf16
      layer's (``moe_oracle.backward``).

    ``quant`` (default :func:`mx_roundtrip`) is the quantise-dequantise round
    trip; with the identity it is the bf16 layer's backward.  ``fwd`` is the
    dict of :func:`forward_mx` (routing and probs).  Returns the dict of
    ``moe_oracle.backward``.
    """
    quant = quant or mx_roundtrip
    x = mo._f64(x); Wr = mo._f64(Wr); W_gu = mo._f64(W_gu); W_down = mo._f64(W_down)
    dY = mo._f64(dY)
    idx = fwd["topk_idx"]; g = fwd["gates"]; real = fwd["real"]
    T, d = x.shape
    E, H2, _ = W_gu.shape
    H = H2 // 2
    k = idx.shape[1]
    Wg, Wu = mo.split_gu(W_gu)
    xq = quant(x)
    dx = np.zeros((T, d))
    dW_gu = np.zeros_like(W_gu)
    dW_down = np.zeros_like(W_down)
    dg = np.zeros((T, k))
    for e in range(E):
        if not (idx == e).any():
            continue
        # expert e's weight operands, quantised once: W_gate, W_up, W_down
        # along their rows (the forward), W_down^T and W_gu^T along the
        # data-gradient products' reduction axes
        qg, qu, qd = quant(Wg[e]), quant(Wu[e]), quant(W_down[e])
        qd_k, qgu_k = roundtrip_k(W_down[e], quant), roundtrip_k(W_gu[e], quant)
        for j in range(k):
            rows = np.nonzero(idx[:, j] == e)[0]
            if not rows.size:
                continue
            where = dict(e=e, j=j, rows=rows)
            a = xq[rows] @ qg.T
            b = xq[rows] @ qu.T
            hf = mo.silu(a) * b
            out = mo._store(rnd, "out", _quantised(rnd, "q_h", hf, quant, where) @ qd.T, where)
            dg[rows, j] = (dY[rows] * out).sum(axis=1)
            h = mo._store(rnd, "h", hf, where)
            # d_out = g dY and d_gu = [da | db] enter their MX products
            # quantised from their own values; their bf16 storage rounding
            # feeds only the weight-gradient products
            d_out_v = g[rows, j][:, None] * dY[rows]
            d_out = mo._store(rnd, "d_out", d_out_v, where)
            dH = _quantised(rnd, "q_d_out", d_out_v, quant, where) @ qd_k
            da_v, db_v = mo.swiglu_backward(dH, _store16(rnd, "a16", a, where),
                                            _store16(rnd, "b16", b, where))
            da, db = mo._store(rnd, "da", da_v, where), mo._store(rnd, "db", db_v, where)
            d_gu = np.concatenate([da_v, db_v], axis=1)
            dx[rows] += mo._store(rnd, "dxe", _quantised(rnd, "q_d_gu", d_gu, quant, where) @ qgu_k,
                                  where)
            dW_down[e] += d_out.T @ h
            dW_gu[e, :H] += da.T @ x[rows]
            dW_gu[e, H:] += db.T @ x[rows]
    # the shared expert, the router and the routing gradient: the bf16 layer's
    dWs_gu = dWs_down = None
    if Ws_gu is not None:
        dxs, dWs_gu, dWs_down = mo.shared_backward(x, Ws_gu, Ws_down, dY, real, rnd)
        dx += dxs
    d_logits = mo.router_logit_grad(dg, idx, g, fwd["probs"], norm_topk)
    d_logits += mo.aux_logit_grad(fwd["probs"], fwd["f"], real, aux_coef)
    if z_coef:
        d_logits += mo.z_logit_grad(fwd["logits"], real, z_coef)
    dx += d_logits @ Wr.T
    dWr = x.T @ d_logits
    return dict(dx=dx, dWr=dWr, dW_gu=dW_gu, dW_down=dW_down, dWs_gu=dWs_gu,
                dWs_down=dWs_down, d_logits=d_logits, dg=dg)


def forward_mx_train(x, Wr, W_gu, W_down, Ws_gu=None, Ws_down=None, k=2, bias=None,
                     valid=None, norm_topk=True, logits=None, rnd=None):
    """The forward of the MXFP8 training step: the routed experts in MXFP8,
    the shared expert in bf16 (:func:`experts_forward_mx` with shared_mx
    False), router and route unchanged."""
    if logits is None:
        logits = mo.router_logits(x, Wr).astype(np.float32)
    r = mo.route(logits, k, bias=bias, valid=valid, norm_topk=norm_topk)
    y, routed = experts_forward_mx(x, r["topk_idx"], r["gates"], W_gu, W_down, Ws_gu,
                                   Ws_down, valid, shared_mx=False, rnd=rnd)
    r.update(y=y, routed=routed, logits=np.asarray(logits))
    return r
