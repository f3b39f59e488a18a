"""CPU fp64 oracle of the sparse Mixture-of-Experts feed-forward layer.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
of ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import or
run this module.  It shares no code with the CUDA path and never imports it.

It is a plain, slow, obviously correct restatement of what the layer
computes, in numpy float64, following these pages:

* "KochiLLM v1.0" model card, Architecture: the MoE FFN applies a shared
  expert to every token plus the top-2 of 4 routed experts, with the gate
  weights renormalised over the selected 2; the loss adds
  0.01 x (E x sum_i f_i p_i) as the load-balancing term.  Configuration:
  the experts are SwiGLU.
* "spark-gpt" README, feature list: bias-free fp32-softmax top-k routing,
  packed SwiGLU experts, selected-probability renormalisation (optional,
  ``--no-norm-topk-prob``), and the auxiliary statistic computed over real
  (non-filler) tokens only.
* "KohakUwULLM" README, Key features: DeepSeekMoE with aux-loss-free load
  balancing, read as a per-expert bias that enters the selection only.

Readings where the pages leave a step open (each one is listed in the design
notes of the repository):

* f_e = counts_e / (k * T_real) and p_e = mean over real tokens of the full,
  unbiased softmax, so sum f = sum p = 1 and E * sum f p = 1 at balance.
* Selection: the k largest keys, equal keys -> the lower expert index first;
  slot order is that ranking (slot 0 = largest key).
* PAD tokens: not routed, not counted, no shared expert; their output and
  their gradients are zero.
* The shared expert is ungated (weight 1); n shared experts of hidden H_s
  are one SwiGLU of hidden n*H_s with concatenated weights.
* Backward: the gradient of  <dY, y> + aux_coef * aux  with the hard counts
  (f) held constant; the selection bias gets no gradient.
* Storage points (the optional hook ``rnd``, see :func:`_store`): the values a
  bf16-storage layer keeps between its products -- h, each routed slot's
  expert output, d_out = g dY, a, b, (da, db) and each routed slot's dx
  contribution -- may be rounded there; without the hook everything is exact.

Weight layouts: W_gu [E][2H][d] (rows [0,H) gate, [H,2H) up),
W_down [E][d][H], Ws_gu [2Hs][d], Ws_down [d][Hs], W_r [d][E].
Parity pins: every function here is pinned by the tests in
``tests/test_oracle_pins.py`` (brute force, closed forms, invariants,
finite differences) and the storage hook by ``tests/test_oracle_storage.py``
(a one-token layer worked out by hand); none is left unpinned.
"""
from __future__ import annotations

import numpy as np

f64 = np.float64


def _np(a):
    """Tensor/array -> numpy, dtype kept (bf16/fp16 widen exactly to fp32)."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch  # CPU tensors only; torch here is plumbing
        t = a.detach().cpu()
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.float()
        return t.numpy()
    return np.asarray(a)


def _f64(a):
    return None if a is None else _np(a).astype(f64)


def sigmoid(a):
    return 1.0 / (1.0 + np.exp(-a))


def silu(a):
    """SiLU (swish) a * sigmoid(a) -- the gate nonlinearity of SwiGLU."""
    return a * sigmoid(a)


# --------------------------------------------------------------------------
# Router ("spark-gpt" README: bias-free router; logits in fp32)
# --------------------------------------------------------------------------

def router_logits(x, Wr):
    """L = x . W_r  (bias-free linear router), exact in fp64."""
    return _f64(x) @ _f64(Wr)


def softmax(L):
    """Row softmax in fp64: exp(L - max) / sum exp(L - max)."""
    L = np.asarray(L, dtype=f64)
    z = np.exp(L - L.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def select_topk(key, k):
    """Indices of the k largest keys per row, largest first; equal keys are
    taken lower index first.  A stable sort on -key keeps equal keys in
    index order (-0.0 and +0.0 compare equal)."""
    key = np.asarray(key)
    order = np.argsort(-key, axis=1, kind="stable")
    return order[:, :k]


def route(logits, k, bias=None, valid=None, norm_topk=True):
    """Top-k routing with renormalised gates and the f.p statistic.

    "KochiLLM v1.0" card, Architecture (top-2 of 4, gates renormalised over
    the selected 2; aux = E * sum_i f_i p_i); "spark-gpt" README feature list
    (fp32-softmax top-k, selected-probability renormalisation, statistic over
    real tokens only).

    logits: [T][E].  float32 logits are the kernel's precision: the selection
    key is formed in fp32 (logits + bias as one fp32 add), so decisions are
    taken in the same precision as on the GPU.  float64 logits keep the key in
    fp64 (used by the finite-difference pins).
    Returns dict: topk_idx [T][k] (-1 on PAD), gates [T][k] (0 on PAD),
    probs [T][E] (full softmax), counts [E], f [E], p [E], aux, T_real.
    """
    L = np.asarray(_np(logits))
    T, E = L.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    if bias is None:
        key = L
    else:
        b = np.asarray(_np(bias))
        key = (L.astype(np.float32) + b.astype(np.float32)) if L.dtype == np.float32 \
            else L + b.astype(f64)
    idx = select_topk(key, k)
    s = softmax(L.astype(f64))
    real = np.ones(T, dtype=bool) if valid is None else (np.asarray(_np(valid)) != 0)
    r = route_stats(s, idx, real, norm_topk)
    r.update(router_metrics(L, r["counts"], real))
    return r


def logsumexp(L):
    """Row log-sum-exp in fp64: max + ln sum exp(L - max)."""
    L = np.asarray(L, dtype=f64)
    m = L.max(axis=-1)
    return m + np.log(np.exp(L - m[..., None]).sum(axis=-1))


def router_metrics(L, counts, real):
    """Routing metrics ("spark-gpt" README: assignment min/max/CV, router
    entropy, unused experts) and the router z-loss ("KohakUwULLM" README,
    Key features: z-loss), read as the mean over real tokens of the squared
    log-sum-exp of the logits.  Entropy in nats of the full softmax, averaged
    over real tokens; CV = population std / mean of the per-expert counts."""
    L = np.asarray(L, dtype=f64)
    counts = np.asarray(counts, dtype=f64)
    Tr = int(np.asarray(real).sum())
    lse = logsumexp(L)
    s = softmax(L)
    with np.errstate(divide="ignore", invalid="ignore"):
        ent = -(s * np.where(s > 0, np.log(s), 0.0)).sum(axis=-1)
    mean = counts.mean()
    return dict(z_loss=float((lse[real] ** 2).mean()) if Tr else 0.0,
                entropy=float(ent[real].mean()) if Tr else 0.0,
                count_min=float(counts.min()), count_max=float(counts.max()),
                count_cv=float(counts.std() / mean) if mean > 0 else 0.0,
                unused=int((counts == 0).sum()), T_real=Tr)


def route_stats(s, idx, real, norm_topk=True):
    """Gates, counts, f, p and aux for a given selection ``idx`` [T][k] of
    the softmax ``s`` [T][E] (PAD rows: real == False)."""
    T, E = s.shape
    k = idx.shape[1]
    idx = np.where(real[:, None], idx, 0)
    sel = np.take_along_axis(s, idx, axis=1)
    gates = sel / sel.sum(axis=1, keepdims=True) if norm_topk else sel.copy()
    idx = np.where(real[:, None], idx, -1).astype(np.int64)
    gates = np.where(real[:, None], gates, 0.0)
    T_real = int(real.sum())
    counts = np.zeros(E, dtype=np.int64)
    for j in range(k):
        counts += np.bincount(idx[real, j], minlength=E)
    if T_real > 0:
        f = counts / f64(k * T_real)
        p = s[real].sum(axis=0) / f64(T_real)
    else:
        f = np.zeros(E)
        p = np.zeros(E)
    aux = f64(E) * float(np.dot(f, p))
    return dict(topk_idx=idx, gates=gates, probs=s, counts=counts, f=f, p=p,
                aux=aux, T_real=T_real, real=real)


# --------------------------------------------------------------------------
# Dispatch: stable counting sort of (token, slot) pairs by expert
# --------------------------------------------------------------------------

def permute(topk_idx, E):
    """Expert-contiguous order of the (t, j) pairs.

    Pairs are keyed q = t*k + j and sorted by expert with a stable sort, so
    each expert's segment lists its tokens in ascending t.  Returns
    offsets [E+1] (exclusive scan of counts), perm [M] (perm[r] = q of row r)
    and inv [T*k] (row of pair q, -1 for PAD tokens).
    """
    idx = np.asarray(topk_idx).reshape(-1)
    q_real = np.nonzero(idx >= 0)[0]
    perm = q_real[np.argsort(idx[q_real], kind="stable")]
    counts = np.bincount(idx[q_real], minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    inv = np.full(idx.shape[0], -1, dtype=np.int64)
    inv[perm] = np.arange(perm.shape[0])
    return offsets, perm.astype(np.int64), inv


# --------------------------------------------------------------------------
# Experts ("KochiLLM v1.0" card: SwiGLU experts, hidden 2 x dim)
# --------------------------------------------------------------------------

def _exact(a):
    return a


def _store(rnd, point, v, where):
    """The value kept at storage point ``point`` ("h", "out", "a", "b",
    "d_out", "da", "db", "dxe"): ``rnd(v)``, or ``rnd.store(point, v, where)`` when the hook
    has that method (``where`` names the rows: expert e, slot j, token rows,
    or shared=True).  No arithmetic happens here."""
    if rnd is None:
        return v
    if hasattr(rnd, "store"):
        return rnd.store(point, v, where)
    return rnd(v)


def swiglu_parts(xr, Wg, Wu, Wd, rnd=None, where=None):
    """One SwiGLU FFN on rows xr: a = xr Wg^T, b = xr Wu^T,
    h = silu(a) * b, out = h Wd^T.  Returns (out, a, b, h).

    ``rnd`` (default: none) rounds the stored hidden h before the down
    projection; it models a storage precision, the arithmetic is unchanged."""
    a = xr @ Wg.T
    b = xr @ Wu.T
    h = _store(rnd, "h", silu(a) * b, where)
    return h @ Wd.T, a, b, h


def swiglu_backward(dh, a, b):
    """Chain rule through h = silu(a) * b: given dh = dJ/dh, returns
    (da, db) = (dh * b * s(a) * (1 + a (1 - s(a))), dh * silu(a)),
    s the logistic sigmoid."""
    sa = sigmoid(a)
    return dh * b * sa * (1.0 + a * (1.0 - sa)), dh * silu(a)


def stored_d_out(g, dY, rnd=None, where=None):
    """d_out = g dY per routed row, as kept between the combine backward and
    the expert products: one storage rounding ``rnd`` of the product (none by
    default)."""
    return _store(rnd, "d_out", g[:, None] * dY, where)


def stored_swiglu_backward(dh, a, b, rnd=None, where=None):
    """(da, db) as kept for the dX and dW products: the chain rule of
    :func:`swiglu_backward` taken on the stored pre-activations rnd(a) and
    rnd(b), and each result stored once more (rnd).  dh itself is not stored:
    it is the dH product's unrounded result."""
    da, db = swiglu_backward(dh, _store(rnd, "a", a, where), _store(rnd, "b", b, where))
    return _store(rnd, "da", da, where), _store(rnd, "db", db, where)


def split_gu(W_gu):
    """[.., 2H, d] packed gate/up -> (gate [.., H, d], up [.., H, d])."""
    H = W_gu.shape[-2] // 2
    return W_gu[..., :H, :], W_gu[..., H:, :]


def experts_forward(x, topk_idx, gates, W_gu, W_down, Ws_gu=None, Ws_down=None,
                    valid=None, rnd=None):
    """y_t = sum_j g_{t,j} F_{e_{t,j}}(x_t) + F_shared(x_t) for real t; PAD -> 0.

    Per token and slot, the expert the router chose is applied (vectorised
    over the tokens that chose the same expert in the same slot, one fp64
    matmul each), then the gated outputs are summed.
    Returns (y [T][d], routed [T][k][d] = F_{e_{t,j}}(x_t)).
    ``rnd`` rounds the stored hidden activations (see :func:`swiglu_parts`)
    and each routed slot's expert output before the gated sum (point "out").
    """
    x = _f64(x); W_gu = _f64(W_gu); W_down = _f64(W_down)
    idx = np.asarray(topk_idx); g = np.asarray(gates, dtype=f64)
    T, d = x.shape
    E = W_gu.shape[0]
    k = idx.shape[1]
    Wg, Wu = split_gu(W_gu)
    routed = np.zeros((T, k, d))
    for j in range(k):
        for e in range(E):
            rows = np.nonzero(idx[:, j] == e)[0]
            if rows.size:
                where = dict(e=e, j=j, rows=rows)
                out, *_ = swiglu_parts(x[rows], Wg[e], Wu[e], W_down[e], rnd, where)
                # each slot's expert output is kept until the slots are summed
                routed[rows, j] = _store(rnd, "out", out, where)
    y = np.einsum("tj,tjd->td", g, routed)
    real = np.ones(T, dtype=bool) if valid is None else (np.asarray(_np(valid)) != 0)
    if Ws_gu is not None:
        sg, su = split_gu(_f64(Ws_gu))
        shared, *_ = swiglu_parts(x[real], sg, su, _f64(Ws_down), rnd,
                                  dict(shared=True, rows=np.nonzero(real)[0]))
        y[real] += shared
    y[~real] = 0.0
    return y, routed


def forward(x, Wr, W_gu, W_down, Ws_gu=None, Ws_down=None, k=2, bias=None,
            valid=None, norm_topk=True, logits=None):
    """Whole layer: router logits -> route -> experts -> combine.

    The routing decision is taken on fp32 logits (the router's precision:
    logits = x . W_r in fp32).  The oracle forms them as the fp32 rounding of
    the exact product unless ``logits`` is given.
    """
    if logits is None:
        logits = router_logits(x, Wr).astype(np.float32)
    r = route(logits, k, bias=bias, valid=valid, norm_topk=norm_topk)
    y, routed = experts_forward(x, r["topk_idx"], r["gates"], W_gu, W_down,
                                Ws_gu, Ws_down, valid)
    r.update(y=y, routed=routed, logits=np.asarray(logits))
    return r


# --------------------------------------------------------------------------
# Backward: gradient of <dY, y> + aux_coef * aux, hard counts held constant
# --------------------------------------------------------------------------

def router_logit_grad(dg, topk_idx, gates, probs, norm_topk):
    """dJ/dL from the gate gradients dg [T][k] (main term).

    With renormalisation the k gates are a softmax over the selected logits,
    so dL_{e_j} = g_j (dg_j - sum_i g_i dg_i) and unselected logits get 0.
    Without it the gates are entries of the full softmax s, so
    dL_e = s_e (u_e - sum_m s_m u_m) with u = dg scattered onto the experts.
    """
    T, k = dg.shape
    E = probs.shape[1]
    dL = np.zeros((T, E))
    real = topk_idx[:, 0] >= 0
    if norm_topk:
        c = (gates * dg).sum(axis=1, keepdims=True)
        contrib = gates * (dg - c)
        for j in range(k):
            rr = np.nonzero(real)[0]
            dL[rr, topk_idx[rr, j]] += contrib[rr, j]
    else:
        u = np.zeros((T, E))
        rr = np.nonzero(real)[0]
        for j in range(k):
            u[rr, topk_idx[rr, j]] += dg[rr, j]
        dL = probs * (u - (probs * u).sum(axis=1, keepdims=True))
        dL[~real] = 0.0
    return dL


def aux_logit_grad(probs, f, real, aux_coef):
    """d(aux_coef * E * sum_e f_e p_e)/dL_{t,e} with f constant:
    (aux_coef * E / T_real) * s_{t,e} * (f_e - sum_i f_i s_{t,i}), real t."""
    T, E = probs.shape
    T_real = int(real.sum())
    out = np.zeros((T, E))
    if T_real == 0:
        return out
    sf = probs @ f
    out = (aux_coef * E / T_real) * probs * (f[None, :] - sf[:, None])
    out[~real] = 0.0
    return out


def z_logit_grad(L, real, z_coef):
    """d(z_coef * mean_real(lse_t^2))/dL_{t,e} = (2 z_coef / T_real) lse_t s_{t,e}."""
    L = np.asarray(L, dtype=f64)
    out = np.zeros_like(L)
    Tr = int(np.asarray(real).sum())
    if Tr == 0 or z_coef == 0:
        return out
    out = (2.0 * z_coef / Tr) * logsumexp(L)[:, None] * softmax(L)
    out[~np.asarray(real)] = 0.0
    return out


def backward(x, Wr, W_gu, W_down, Ws_gu, Ws_down, fwd, dY, norm_topk=True,
             aux_coef=0.01, rnd=None, z_coef=0.0):
    """Gradients of J = <dY, y> + aux_coef * aux + z_coef * z_loss by the
    chain rule (z_loss needs fwd["logits"] when z_coef is non-zero).

    ``fwd`` is the dict returned by :func:`forward` (routing and probs).
    Returns dict: dx [T][d], dWr [d][E], dW_gu [E][2H][d], dW_down [E][d][H],
    dWs_gu, dWs_down (or None), d_logits [T][E], dg [T][k].

    ``rnd`` (default: none) rounds the values a bf16-storage implementation
    keeps between its matrix products (see :func:`_store` for a hook that
    also receives the storage point and rows) -- the hidden h
    (:func:`swiglu_parts`), each routed slot's expert output ("out", read
    for dg), d_out = g dY of the routed rows (:func:`stored_d_out`), the
    saved pre-activations a and b and the results (da, db) of the SwiGLU
    chain rule (:func:`stored_swiglu_backward`), and each routed slot's dx
    contribution before the slots are summed ("dxe") -- without changing any
    arithmetic step.
    The shared expert's d_out is dY itself (an input, not rounded again).
    With ``rnd`` None this is the exact gradient.
    """
    x = _f64(x); Wr = _f64(Wr); W_gu = _f64(W_gu); W_down = _f64(W_down)
    dY = _f64(dY)
    idx = fwd["topk_idx"]; g = fwd["gates"]; real = fwd["real"]
    T, d = x.shape
    E, H2, _ = W_gu.shape
    H = H2 // 2
    k = idx.shape[1]
    Wg, Wu = split_gu(W_gu)
    dx = np.zeros((T, d))
    dW_gu = np.zeros_like(W_gu)
    dW_down = np.zeros_like(W_down)
    dg = np.zeros((T, k))

    for j in range(k):
        for e in range(E):
            rows = np.nonzero(idx[:, j] == e)[0]
            if not rows.size:
                continue
            xr = x[rows]
            where = dict(e=e, j=j, rows=rows)
            out, a, b, h = swiglu_parts(xr, Wg[e], Wu[e], W_down[e], rnd, where)
            out = _store(rnd, "out", out, where)
            dg[rows, j] = (dY[rows] * out).sum(axis=1)
            d_out = stored_d_out(g[rows, j], dY[rows], rnd, where)
            da, db = stored_swiglu_backward(d_out @ W_down[e], a, b, rnd, where)
            # the slot's dx contribution is kept until the slots are summed
            dx[rows] += _store(rnd, "dxe", da @ Wg[e] + db @ Wu[e], where)
            dW_down[e] += d_out.T @ h
            dW_gu[e, :H] += da.T @ xr
            dW_gu[e, H:] += db.T @ xr
    dWs_gu = dWs_down = None
    if Ws_gu is not None:
        dxs, dWs_gu, dWs_down = shared_backward(x, Ws_gu, Ws_down, dY, real, rnd)
        dx += dxs
    d_logits = router_logit_grad(dg, idx, g, fwd["probs"], norm_topk)
    d_logits += aux_logit_grad(fwd["probs"], fwd["f"], real, aux_coef)
    if z_coef:
        d_logits += z_logit_grad(fwd["logits"], real, z_coef)
    dx += d_logits @ Wr.T
    dWr = x.T @ d_logits
    return dict(dx=dx, dWr=dWr, dW_gu=dW_gu, dW_down=dW_down, dWs_gu=dWs_gu,
                dWs_down=dWs_down, d_logits=d_logits, dg=dg)


def shared_backward(x, Ws_gu, Ws_down, dY, real, rnd=None):
    """The shared expert's part of the backward: its SwiGLU on the real
    tokens (weight 1), d_out = dY itself.  Returns (dx contribution [T][d],
    dWs_gu, dWs_down); storage points through ``rnd`` as in :func:`backward`."""
    x = _f64(x); dY = _f64(dY)
    Ws_gu_ = _f64(Ws_gu); Ws_down_ = _f64(Ws_down)
    sg, su = split_gu(Ws_gu_)
    rows = np.nonzero(real)[0]
    xr = x[rows]
    where = dict(shared=True, rows=rows)
    out, a, b, h = swiglu_parts(xr, sg, su, Ws_down_, rnd, where)
    da, db = stored_swiglu_backward(dY[rows] @ Ws_down_, a, b, rnd, where)
    dx = np.zeros_like(x)
    dx[rows] = da @ sg + db @ su
    Hs = sg.shape[0]
    dWs_gu = np.zeros_like(Ws_gu_)
    dWs_gu[:Hs] = da.T @ xr
    dWs_gu[Hs:] = db.T @ xr
    dWs_down = dY[rows].T @ h
    return dx, dWs_gu, dWs_down


def objective(x, Wr, W_gu, W_down, Ws_gu, Ws_down, dY, k, bias=None, valid=None,
              norm_topk=True, aux_coef=0.01, counts_f=None, z_coef=0.0):
    """J = <dY, y> + aux_coef * aux + z_coef * z_loss with fp64 logits
    (finite-difference pins).

    ``counts_f`` holds f fixed (the hard counts are not differentiated).
    """
    L = router_logits(x, Wr)
    r = route(L, k, bias=bias, valid=valid, norm_topk=norm_topk)
    y, _ = experts_forward(x, r["topk_idx"], r["gates"], W_gu, W_down, Ws_gu,
                           Ws_down, valid)
    f = r["f"] if counts_f is None else counts_f
    aux = r["probs"].shape[1] * float(np.dot(f, r["p"]))
    return float((_f64(dY) * y).sum()) + aux_coef * aux + z_coef * r["z_loss"], r
