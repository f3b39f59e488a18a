"""Why the GPU tests compare gradients with the storage-rounded oracle (CPU only).

The layer stores its GEMM operands in bf16 (hidden h, saved pre-activations,
d_out = g dY, (da, db)); tensor cores take bf16 operands.  Even an ideal
pipeline with exact accumulation and rounding only at those storage points
misses a max normalised error of 1e-2 against the exact gradient on the
expert weight gradients of the many-expert shapes, while its
Frobenius-relative error stays near 2e-3.  So the GPU tests hold every bf16
output and gradient to max normalised |gpu - ideal| <= 1e-2, where ideal is
the oracle with the same storage rounding (the hook pinned in
test_oracle_storage.py), and to Frobenius-relative |gpu - exact| <= 1e-2.
"""
import numpy as np

from mixture_experts_ffn_02_gb300 import synth
from oracle import moe_oracle as O
from moe_check import bf16_round, frob_err, norm_err


def test_ideal_bf16_storage_exceeds_literal_max_metric_on_weight_grads():
    s = synth.scaled(synth.shape(4), T=300, T_real=None, zipf_bias=0.0)
    inp = synth.make_inputs(s, seed=0, with_grad=True)
    fwd = O.forward(inp["x"], inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"],
                    inp["Ws_down"], k=s.k)
    args = (inp["x"], inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"], inp["Ws_down"],
            fwd, inp["dY"])
    exact = O.backward(*args)
    ideal = O.backward(*args, rnd=bf16_round)
    worst = max(norm_err(ideal[n], exact[n]) for n in ("dW_gu", "dW_down"))
    assert worst > 1e-2
    for n in ("dW_gu", "dW_down", "dx", "d_logits", "dWr"):
        assert frob_err(ideal[n], exact[n]) < 5e-3, n


def test_storage_rounding_hook_is_identity_when_absent():
    s = synth.scaled(synth.shape(1), T=40)
    inp = synth.make_inputs(s, seed=1, with_grad=True)
    fwd = O.forward(inp["x"], inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"],
                    inp["Ws_down"], k=s.k)
    args = (inp["x"], inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"], inp["Ws_down"],
            fwd, inp["dY"])
    a = O.backward(*args)
    b = O.backward(*args, rnd=lambda v: v)
    for n in a:
        if a[n] is not None:
            np.testing.assert_array_equal(a[n], b[n])
    # with bf16 storage the stored hidden is exactly bf16(h)
    xr = np.asarray(inp["x"].double())
    Wg, Wu = O.split_gu(inp["W_gu"].double().numpy()[0])
    _, a_, b_, h_ = O.swiglu_parts(xr, Wg, Wu, inp["W_down"].double().numpy()[0], bf16_round)
    np.testing.assert_array_equal(h_, bf16_round(O.silu(a_) * b_))


class _FlipSome:
    """Storage rounding to bf16 that stores the other bf16 neighbour at a
    seeded fraction of the elements of h -- what a pipeline whose fp32 h
    differs from the exact one by a few fp32 ulps does near rounding
    boundaries (the GPU's rate is about 1e-3)."""

    def __init__(self, frac, seed=0):
        self.frac = frac
        self.rng = np.random.default_rng(seed)

    def store(self, point, v, where):
        r = bf16_round(v)
        if point != "h":
            return r
        flip = self.rng.random(r.shape) < self.frac
        a = np.abs(r)
        ulp = np.where(a > 0, np.exp2(np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7), 0.0)
        return np.where(flip, r + np.where(v >= r, ulp, -ulp), r)


def test_one_ulp_flips_of_stored_h_exceed_max_metric_on_weight_grads():
    """Why the GPU tests continue the oracle from the GPU's own stored value
    where it took the other rounding (moe_check.AdoptStored): one-ulp flips
    of 0.1% of the stored hidden h, every one of them a correct rounding of
    a value a few fp32 ulps away from the exact one, already move the
    max-normalised weight gradient by more than 1e-2 on the 128-expert shape,
    while its Frobenius-relative change stays near 1e-4."""
    s = synth.scaled(synth.shape(5), T=160, T_real=None)
    inp = synth.make_inputs(s, seed=0, with_grad=True)
    fwd = O.forward(inp["x"], inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"],
                    inp["Ws_down"], k=s.k)
    args = (inp["x"], inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"], inp["Ws_down"],
            fwd, inp["dY"])
    ideal = O.backward(*args, rnd=bf16_round)
    flipped = O.backward(*args, rnd=_FlipSome(1e-3))
    assert norm_err(flipped["dW_down"], ideal["dW_down"]) > 1e-2
    assert frob_err(flipped["dW_down"], ideal["dW_down"]) < 1e-3


def test_mx_valid_accepts_exactly_the_nearby_quantisations():
    """moe_check.mx_valid, which lets the GPU tests continue from the GPU's
    own MX codes: the oracle's codes are valid and not "other"; the other
    e4m3 neighbour is valid only where v lies within the fp32 tolerance of
    the midpoint between the two; a code two steps away, or a block scale
    one off away from a power of two, is invalid."""
    from moe_check import mx_valid
    from oracle import mx_oracle as M
    rng = np.random.default_rng(3)
    v = rng.standard_normal((4, 64))
    c, s = M.mx_quantize(v)
    ok, other = mx_valid(v, c, s)
    assert ok.all() and not other.any()
    # put element (0, 5) on the midpoint between two codes of its block grid
    X = s[0, 0].astype(float) - 127
    g = M.e4m3_decode(c[0, 5]) * 2.0 ** X
    up = M.e4m3_decode(np.uint8(c[0, 5] + 1)) * 2.0 ** X
    v2 = v.copy()
    v2[0, 5] = (g + up) / 2 * (1 + 2.0 ** -30)       # just above the midpoint
    c2, s2 = M.mx_quantize(v2)
    assert s2[0, 0] == s[0, 0]
    flip = c2.copy()
    flip[0, 5] = c2[0, 5] - 1                         # the neighbour below: valid here
    ok, other = mx_valid(v2, flip, s2)
    assert ok.all() and other.sum() == 1
    flip = c.copy()
    flip[1, 7] = c[1, 7] + 1 if c[1, 7] & 0x7F < 0x7D else c[1, 7] - 1    # far from a midpoint
    ok, _ = mx_valid(v, flip, s)
    assert (~ok).sum() == 1 and not ok[1, 7]
    two = c.copy()
    two[2, 3] = (c[2, 3] & 0x80) | max((c[2, 3] & 0x7F) - 2, 0)
    ok, _ = mx_valid(v, two, s)
    assert not ok[2, 3]
    bad_s = s.copy()
    bad_s[3, 1] += 1
    amax = np.abs(v[3, 32:64]).max()
    assert abs(np.log2(amax) - np.round(np.log2(amax))) > 1e-3   # not near a power of two
    ok, _ = mx_valid(v, c, bad_s)
    assert not ok[3, 32:64].any() and ok[3, :32].all()


def test_fp16_neighbours_bracket_and_adopt():
    """moe_check.fp16_neighbours: the rounding and the other neighbour of v
    bracket it, one binary16 ulp apart (also across a binade edge), and an
    AdoptStored point named *16 takes either without counting it invalid."""
    from moe_check import AdoptStored, fp16_neighbours
    v = np.array([1 + 2.0 ** -12, 2 - 2.0 ** -13, -3.3, 1e-6, 700.1])
    r, other, _ = fp16_neighbours(v)
    assert ((np.minimum(r, other) <= v) & (v <= np.maximum(r, other))).all()
    assert r[1] == 2.0 and other[1] == 2 - 2.0 ** -10       # ulp 2^-10 below 2
    ad = AdoptStored({}, np.zeros(1, int), 1)
    ad.adopt("a16", v, other)
    ad.adopt("a16", v, r)
    n, diff, bad = ad.stats["a16"]
    assert (n, diff, bad) == (10, 5, 0)
    ad.adopt("a16", v, r + 4 * np.abs(other - r))
    assert ad.stats["a16"][2] > 0
