"""Pins for the CPU oracle: values and laws fixed by the pages and by the
mathematics, independent of the oracle's own code path.

Each test names what it pins.  A plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand, a wrong tie rule, a wrong
normalisation of f or p) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- selection

@pytest.mark.parametrize("E,k", [(3, 1), (4, 2), (5, 3), (6, 2), (6, 5), (4, 4)])
def test_selection_brute_force(E, k):
    """Top-k by enumerating every k-subset: the selected set has the largest
    key sum; among equal sums the lexicographically smallest index set wins
    (= lower index wins ties).  Keys are small integers, so sums are exact and
    ties are frequent.  Slot order: larger key first, equal keys by index."""
    rng = _rng(E * 10 + k)
    key = rng.integers(-3, 4, size=(300, E)).astype(np.float32)
    got = O.select_topk(key, k)
    for t in range(key.shape[0]):
        best = None
        for sub in itertools.combinations(range(E), k):
            sc = float(sum(key[t, list(sub)]))
            if best is None or sc > best[0] or (sc == best[0] and sub < best[1]):
                best = (sc, sub)
        assert sorted(got[t].tolist()) == list(best[1])
        slots = got[t].tolist()
        for a, b in zip(slots, slots[1:]):
            assert key[t, a] > key[t, b] or (key[t, a] == key[t, b] and a < b)


def test_signed_zero_is_a_tie():
    key = np.array([[0.0, -0.0, -1.0], [-0.0, 0.0, -1.0]], dtype=np.float32)
    assert O.select_topk(key, 1)[:, 0].tolist() == [0, 0]


def test_equal_logits_tie_rule_and_balance():
    """Equal logits: p_e = 1/E exactly; every token picks experts 0..k-1, so
    f = 1/k on those and 0 elsewhere; aux = E * sum f p = 1."""
    T, E, k = 64, 8, 3
    r = O.route(np.zeros((T, E), np.float32), k)
    assert (r["topk_idx"] == np.arange(k)).all()
    np.testing.assert_array_equal(r["p"], np.full(E, 1.0 / E))
    np.testing.assert_array_equal(r["f"][:k], np.full(k, 1.0 / k))
    assert (r["f"][k:] == 0).all()
    assert r["aux"] == pytest.approx(1.0, abs=1e-15)
    np.testing.assert_allclose(r["gates"], 1.0 / k, rtol=0, atol=1e-15)
    r2 = O.route(np.zeros((T, E), np.float32), k, norm_topk=False)
    np.testing.assert_allclose(r2["gates"], 1.0 / E, rtol=0, atol=1e-15)


def test_router_metrics_closed_forms():
    """Equal logits c: logsumexp = c + ln E, so z_loss = (c + ln E)^2; the
    entropy is ln E (its maximum); experts 0..k-1 take every token, so
    counts = [T]*k + [0]*(E-k): min 0, max T, E-k unused, CV = sqrt(E/k - 1)."""
    T, E, k, c = 50, 8, 3, 0.75
    r = O.route(np.full((T, E), c, np.float32), k)
    assert r["z_loss"] == pytest.approx((c + math.log(E)) ** 2, rel=1e-12)
    assert r["entropy"] == pytest.approx(math.log(E), rel=1e-12)
    assert (r["count_min"], r["count_max"], r["unused"]) == (0.0, float(T), E - k)
    assert r["count_cv"] == pytest.approx(math.sqrt(E / k - 1), rel=1e-12)
    # a dominant logit: entropy -> 0, logsumexp -> that logit
    L = np.zeros((4, E)); L[:, 2] = 60.0
    r = O.route(L, 1)
    assert r["entropy"] < 1e-20 and r["z_loss"] == pytest.approx(3600.0, rel=1e-12)
    # PAD rows do not count
    valid = np.array([1, 1, 0, 0], np.uint8)
    L2 = np.array([[0.0] * E, [math.log(2.0)] + [0.0] * (E - 1), [9.0] * E, [5.0] * E])
    r = O.route(L2, 2, valid=valid)
    lse = [math.log(E), math.log(E + 1.0)]
    assert r["z_loss"] == pytest.approx((lse[0] ** 2 + lse[1] ** 2) / 2, rel=1e-12)
    assert r["T_real"] == 2


def test_softmax_closed_form():
    """softmax(0, ln 2, ln 3) = (1/6, 2/6, 3/6)."""
    s = O.softmax(np.array([[0.0, math.log(2.0), math.log(3.0)]]))
    np.testing.assert_allclose(s[0], [1 / 6, 2 / 6, 3 / 6], rtol=1e-15)
    # shift invariance with huge logits (no overflow)
    s2 = O.softmax(np.array([[1000.0, 1000.0 + math.log(2.0), 1000.0 + math.log(3.0)]]))
    np.testing.assert_allclose(s2[0], [1 / 6, 2 / 6, 3 / 6], rtol=1e-12)


def test_gates_renorm_and_raw():
    """Renormalised gates sum to 1 and keep the ratios of the selected
    probabilities; without renormalisation the gates are the probabilities."""
    L = O.router_logits(torch.randn(50, 16).bfloat16(), torch.randn(16, 6) * 0.5)
    L32 = L.astype(np.float32)
    r = O.route(L32, 3)
    np.testing.assert_allclose(r["gates"].sum(1), 1.0, atol=1e-15)
    r2 = O.route(L32, 3, norm_topk=False)
    sel = np.take_along_axis(r2["probs"], r2["topk_idx"], 1)
    np.testing.assert_array_equal(r2["gates"], sel)
    np.testing.assert_allclose(r["gates"] * sel.sum(1, keepdims=True), sel, rtol=1e-14)


def test_aux_closed_form_all_to_one_expert():
    """E=2, k=1, every token sends to expert 0 with s = (a, 1-a):
    f = (1, 0), p = (a, 1-a), aux = 2a."""
    a = 0.8
    L = np.tile(np.array([[math.log(a), math.log(1 - a)]]), (10, 1))
    r = O.route(L, 1)
    np.testing.assert_allclose(r["f"], [1.0, 0.0])
    np.testing.assert_allclose(r["p"], [a, 1 - a], rtol=1e-14)
    assert r["aux"] == pytest.approx(2 * a, rel=1e-14)


def test_aux_statistic_sums_and_random_balance():
    """sum f = sum p = 1; with i.i.d. logits E[f_e] = 1/E (5 sigma)."""
    T, E, k = 20000, 8, 2
    L = _rng(3).standard_normal((T, E)).astype(np.float32)
    r = O.route(L, k)
    assert r["f"].sum() == pytest.approx(1.0, abs=1e-12)
    assert r["p"].sum() == pytest.approx(1.0, abs=1e-12)
    assert r["counts"].sum() == T * k
    sigma = math.sqrt((1 / E) * (1 - 1 / E) / (T * k))
    assert np.abs(r["f"] - 1 / E).max() < 5 * sigma * 2  # pairs within a token correlate
    assert np.abs(r["p"] - 1 / E).max() < 0.01


def test_pad_tokens_excluded():
    """PAD rows: not routed (-1), zero gates, not counted; f, p use T_real."""
    T, E, k = 40, 4, 2
    L = _rng(4).standard_normal((T, E)).astype(np.float32)
    valid = np.ones(T, np.uint8)
    valid[30:] = 0
    r = O.route(L, k, valid=valid)
    r_real = O.route(L[:30], k)
    assert (r["topk_idx"][30:] == -1).all() and (r["gates"][30:] == 0).all()
    np.testing.assert_array_equal(r["counts"], r_real["counts"])
    np.testing.assert_allclose(r["p"], r_real["p"], rtol=1e-15)
    assert r["aux"] == pytest.approx(r_real["aux"], rel=1e-15)
    assert r["T_real"] == 30


def test_bias_enters_selection_only():
    """Selection bias changes which experts are chosen, but the gates are the
    unbiased softmax renormalised over the chosen set, and p is unbiased."""
    T, E, k = 100, 6, 2
    L = _rng(5).standard_normal((T, E)).astype(np.float32)
    b = np.array([-1.1 * math.log(e + 1) for e in range(E)], np.float32)
    r = O.route(L, k, bias=b)
    key = L + b
    np.testing.assert_array_equal(r["topk_idx"], O.select_topk(key, k))
    sel = np.take_along_axis(O.softmax(L.astype(np.float64)), r["topk_idx"], 1)
    np.testing.assert_allclose(r["gates"], sel / sel.sum(1, keepdims=True), rtol=1e-14)
    np.testing.assert_allclose(r["p"], O.softmax(L.astype(np.float64)).mean(0), rtol=1e-14)


# ---------------------------------------------------------------- permute

def test_permute_invariants_and_brute_force():
    T, E, k = 97, 5, 3
    L = _rng(6).standard_normal((T, E)).astype(np.float32)
    valid = (_rng(7).random(T) > 0.2).astype(np.uint8)
    r = O.route(L, k, valid=valid)
    offsets, perm, inv = O.permute(r["topk_idx"], E)
    M = int(valid.sum()) * k
    assert offsets[0] == 0 and offsets[-1] == M == perm.shape[0]
    np.testing.assert_array_equal(np.diff(offsets), r["counts"])
    # bijection onto the real pairs, inv o perm = id
    assert sorted(perm.tolist()) == sorted(np.nonzero(r["topk_idx"].reshape(-1) >= 0)[0].tolist())
    np.testing.assert_array_equal(inv[perm], np.arange(M))
    assert (inv[r["topk_idx"].reshape(-1) < 0] == -1).all()
    # brute force: nested loops, expert-major, tokens ascending
    expect = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if r["topk_idx"][t, j] == e:
                    expect.append(t * k + j)
    np.testing.assert_array_equal(perm, expect)
    # each segment holds only its expert
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (r["topk_idx"].reshape(-1)[seg] == e).all()


# ---------------------------------------------------------------- experts

def test_swiglu_closed_form_scalars():
    """d = H = 1, unit weights: F(x) = silu(x) * x;
    silu(1) = 1/(1+e^-1) = 0.7310585786300049, silu(2)*2 = 3.523188311911529."""
    one = np.ones((1, 1))
    out1, *_ = O.swiglu_parts(np.array([[1.0]]), one, one, one)
    out2, *_ = O.swiglu_parts(np.array([[2.0]]), one, one, one)
    assert out1[0, 0] == pytest.approx(0.7310585786300049, rel=1e-15)
    assert out2[0, 0] == pytest.approx(3.523188311911529, rel=1e-15)
    # gate and up are not interchangeable: silu(2x)*x vs silu(x)*2x
    out3, *_ = O.swiglu_parts(np.array([[1.0]]), 2 * one, one, one)
    assert out3[0, 0] == pytest.approx(2.0 / (1.0 + math.exp(-2.0)) * 1.0, rel=1e-15)


def _dense_swiglu_torch(x, Wg, Wu, Wd):
    x, Wg, Wu, Wd = (torch.as_tensor(np.asarray(a, np.float64)) for a in (x, Wg, Wu, Wd))
    return (torch.nn.functional.silu(x @ Wg.T) * (x @ Wu.T) @ Wd.T).numpy()


def test_k_equals_E_identical_experts_is_dense_ffn():
    """k = E with identical experts and renormalised gates: y = F(x) + F_s(x)
    (gates sum to 1), checked against torch fp64 silu/matmul."""
    T, d, E, H, Hs = 33, 16, 4, 24, 8
    g = torch.Generator().manual_seed(11)
    x = torch.randn(T, d, generator=g).bfloat16()
    Wr = torch.randn(d, E, generator=g)
    w1 = torch.randn(2 * H, d, generator=g).bfloat16() * 0.2
    w2 = torch.randn(d, H, generator=g).bfloat16() * 0.2
    W_gu = w1.unsqueeze(0).repeat(E, 1, 1)
    W_down = w2.unsqueeze(0).repeat(E, 1, 1)
    Ws_gu = torch.randn(2 * Hs, d, generator=g).bfloat16() * 0.2
    Ws_down = torch.randn(d, Hs, generator=g).bfloat16() * 0.2
    r = O.forward(x, Wr, W_gu, W_down, Ws_gu, Ws_down, k=E)
    xf = x.double().numpy()
    ref = _dense_swiglu_torch(xf, w1[:H].double(), w1[H:].double(), w2.double()) + \
        _dense_swiglu_torch(xf, Ws_gu[:Hs].double(), Ws_gu[Hs:].double(), Ws_down.double())
    np.testing.assert_allclose(r["y"], ref, rtol=1e-12, atol=1e-12)


def test_dense_masked_brute_force():
    """y_t = sum_e 1[e selected] g_{t,e} F_e(x_t) + F_s(x_t), every expert on
    every token in plain loops: independent of the oracle's gather order."""
    T, d, E, k, H, Hs = 19, 8, 5, 2, 12, 6
    g = torch.Generator().manual_seed(12)
    x = torch.randn(T, d, generator=g).bfloat16()
    Wr = torch.randn(d, E, generator=g)
    W_gu = torch.randn(E, 2 * H, d, generator=g).bfloat16() * 0.3
    W_down = torch.randn(E, d, H, generator=g).bfloat16() * 0.3
    Ws_gu = torch.randn(2 * Hs, d, generator=g).bfloat16() * 0.3
    Ws_down = torch.randn(d, Hs, generator=g).bfloat16() * 0.3
    valid = np.ones(T, np.uint8)
    valid[[3, 17]] = 0
    r = O.forward(x, Wr, W_gu, W_down, Ws_gu, Ws_down, k=k, valid=valid)
    xf = x.double().numpy()
    Wgu = W_gu.double().numpy(); Wd = W_down.double().numpy()
    Sgu = Ws_gu.double().numpy(); Sd = Ws_down.double().numpy()
    for t in range(T):
        if not valid[t]:
            assert (r["y"][t] == 0).all()
            continue
        acc = np.zeros(d)
        for e in range(E):
            w = 0.0
            for j in range(k):
                if r["topk_idx"][t, j] == e:
                    w = r["gates"][t, j]
            a = Wgu[e, :H] @ xf[t]
            b = Wgu[e, H:] @ xf[t]
            acc += w * (Wd[e] @ (a / (1 + np.exp(-a)) * b))
        a = Sgu[:Hs] @ xf[t]
        b = Sgu[Hs:] @ xf[t]
        acc += Sd @ (a / (1 + np.exp(-a)) * b)
        np.testing.assert_allclose(r["y"][t], acc, rtol=1e-12, atol=1e-13)


def test_shared_experts_concatenate():
    """n shared SwiGLU experts of hidden H_s = one SwiGLU of hidden n*H_s with
    gate rows, up rows and down columns concatenated."""
    d, Hs, n = 8, 5, 3
    rng = _rng(13)
    x = rng.standard_normal((7, d))
    parts = [(rng.standard_normal((Hs, d)), rng.standard_normal((Hs, d)),
              rng.standard_normal((d, Hs))) for _ in range(n)]
    tot = sum(O.swiglu_parts(x, *p)[0] for p in parts)
    Wg = np.concatenate([p[0] for p in parts]); Wu = np.concatenate([p[1] for p in parts])
    Wd = np.concatenate([p[2] for p in parts], axis=1)
    np.testing.assert_allclose(O.swiglu_parts(x, Wg, Wu, Wd)[0], tot, rtol=1e-12)


# ---------------------------------------------------------------- shapes

def _layer_params(dim, layers, q, kv, hd, vocab, experts_counted, hidden, router_E,
                  n_embed_mats):
    """Parameter count of a decoder whose experts are three d x H matrices
    (the oracle's W_gu [2H][d] + W_down [d][H])."""
    W_gu = np.empty((2 * hidden, dim)); W_down = np.empty((dim, hidden))
    per_expert = W_gu.size + W_down.size
    attn = dim * q * hd + 2 * dim * kv * hd + q * hd * dim + 2 * hd
    per_layer = attn + 2 * dim + dim * router_E + experts_counted * per_expert
    return layers * per_layer + n_embed_mats * vocab * dim + dim


def test_parameter_counts_pin_expert_shape():
    facts = json.load(open(os.path.join(GOLDEN, "page_facts.json")))
    s = facts["spark_gpt_moe"]
    total = _layer_params(s["dim"], s["layers"], s["q_heads"], s["kv_heads"], s["head_dim"],
                          s["vocab"], s["experts"], s["moe_intermediate"], s["experts"], 2)
    active = _layer_params(s["dim"], s["layers"], s["q_heads"], s["kv_heads"], s["head_dim"],
                           s["vocab"], s["top_k"], s["moe_intermediate"], s["experts"], 2)
    assert abs(total / s["total_params_about"] - 1) < 0.005
    assert abs(active / s["active_params_about"] - 1) < 0.002
    # compute-matched: top-2 x 768 = dense 1536
    assert s["top_k"] * s["moe_intermediate"] == s["dense_intermediate"]
    kc = facts["kochillm"]
    active_k = _layer_params(kc["dim"], kc["layers"], kc["q_heads"], kc["kv_heads"],
                             kc["head_dim"], kc["vocab"], kc["top_k"] + kc["shared_experts"],
                             kc["expert_hidden"], kc["routed_experts"], 1)
    assert abs(active_k / kc["active_params"] - 1) < 5e-4
    assert kc["expert_hidden"] == 2 * kc["dim"]
    assert kc["aux_expert_factor"] == kc["routed_experts"]


# ---------------------------------------------------------------- backward

def _fd_case(seed, T=12, d=8, E=4, k=2, H=6, Hs=4, pad=True, bias=False):
    """Inputs whose routing margins are wide enough that +-eps never flips a
    selection."""
    for s in range(seed, seed + 200):
        rng = _rng(s)
        x = rng.standard_normal((T, d))
        Wr = rng.standard_normal((d, E)) * 0.6
        b = np.array([-0.7 * math.log(e + 1) for e in range(E)]) if bias else None
        key = x @ Wr + (0 if b is None else b)
        srt = np.sort(key, axis=1)[:, ::-1]
        if (srt[:, k - 1] - srt[:, k]).min() > 1e-3:
            break
    W_gu = rng.standard_normal((E, 2 * H, d)) * 0.4
    W_down = rng.standard_normal((E, d, H)) * 0.4
    Ws_gu = rng.standard_normal((2 * Hs, d)) * 0.4 if Hs else None
    Ws_down = rng.standard_normal((d, Hs)) * 0.4 if Hs else None
    dY = rng.standard_normal((T, d))
    valid = None
    if pad:
        valid = np.ones(T, np.uint8)
        valid[[2, T - 1]] = 0
    return dict(x=x, Wr=Wr, W_gu=W_gu, W_down=W_down, Ws_gu=Ws_gu, Ws_down=Ws_down,
                dY=dY, valid=valid, bias=b)


@pytest.mark.parametrize("norm_topk,pad,bias,Hs,zc", [(True, True, False, 4, 0.0),
                                                      (False, True, False, 4, 0.0),
                                                      (True, False, True, 0, 0.0),
                                                      (False, False, True, 3, 0.0),
                                                      (True, True, False, 4, 0.23)])
def test_backward_matches_central_differences(norm_topk, pad, bias, Hs, zc):
    """Every gradient (x, W_r, expert and shared weights, router logits) of
    J = <dY, y> + a * aux + z * z_loss against central differences in fp64."""
    c = _fd_case(21, pad=pad, bias=bias, Hs=Hs)
    k, alpha = 2, 0.37
    L = O.router_logits(c["x"], c["Wr"])
    fwd = O.forward(c["x"], c["Wr"], c["W_gu"], c["W_down"], c["Ws_gu"], c["Ws_down"], k=k,
                    bias=c["bias"], valid=c["valid"], norm_topk=norm_topk, logits=L)
    grads = O.backward(c["x"], c["Wr"], c["W_gu"], c["W_down"], c["Ws_gu"], c["Ws_down"],
                       fwd, c["dY"], norm_topk=norm_topk, aux_coef=alpha, z_coef=zc)
    f0 = fwd["f"]

    def J(**over):
        a = {**c, **over}
        return O.objective(a["x"], a["Wr"], a["W_gu"], a["W_down"], a["Ws_gu"], a["Ws_down"],
                           a["dY"], k, bias=a["bias"], valid=a["valid"], norm_topk=norm_topk,
                           aux_coef=alpha, counts_f=f0, z_coef=zc)[0]

    eps = 1e-6
    rng = _rng(99)
    names = [("x", "dx"), ("Wr", "dWr"), ("W_gu", "dW_gu"), ("W_down", "dW_down")]
    if Hs:
        names += [("Ws_gu", "dWs_gu"), ("Ws_down", "dWs_down")]
    for pname, gname in names:
        P = c[pname]
        flat = rng.choice(P.size, size=min(P.size, 40), replace=False)
        for i in flat:
            ii = np.unravel_index(i, P.shape)
            Pp = P.copy(); Pp[ii] += eps
            Pm = P.copy(); Pm[ii] -= eps
            fd = (J(**{pname: Pp}) - J(**{pname: Pm})) / (2 * eps)
            assert grads[gname][ii] == pytest.approx(fd, rel=1e-6, abs=1e-7), (pname, ii)

    # the logit gradient: differentiate J through the logits directly
    def JL(Lp):
        r = O.route(Lp, k, bias=c["bias"], valid=c["valid"], norm_topk=norm_topk)
        y, _ = O.experts_forward(c["x"], r["topk_idx"], r["gates"], c["W_gu"], c["W_down"],
                                 c["Ws_gu"], c["Ws_down"], c["valid"])
        return (float((c["dY"] * y).sum()) + alpha * L.shape[1] * float(np.dot(f0, r["p"]))
                + zc * r["z_loss"])

    for t in range(L.shape[0]):
        for e in range(L.shape[1]):
            Lp = L.copy(); Lp[t, e] += eps
            Lm = L.copy(); Lm[t, e] -= eps
            fd = (JL(Lp) - JL(Lm)) / (2 * eps)
            assert grads["d_logits"][t, e] == pytest.approx(fd, rel=1e-6, abs=1e-8), (t, e)
    if pad:
        assert (grads["dx"][c["valid"] == 0] == 0).all()
        assert (grads["d_logits"][c["valid"] == 0] == 0).all()
