"""Helpers shared by the GPU parity tests: running the C-ABI layer on seeded
inputs and comparing it with the CPU oracle.

Tolerances:
* routing indices, counts, offsets and the permutation: bit for bit;
* fp32 statistics (f, p, aux), on the same fp32 logits: relative 1e-5;
* bf16 outputs (y) and every gradient, two bounds at once:
    max_i |gpu_i - ideal_i| / RMS(ideal) <= 1e-2, where ``ideal`` is the
    oracle with bf16 rounding at the layer's storage points (the hidden h,
    the saved pre-activations a and b, d_out = g dY, and (da, db)) and exact
    arithmetic otherwise.  When the GPU value is itself stored in bf16, half
    a bf16 ulp of the stored value -- the largest error its own final
    rounding can make -- is taken off each difference first.
    ||gpu - exact||_F / ||exact||_F <= 1e-2 against the exact oracle.
  The plain max|gpu - exact| / RMS(exact) and max|gpu - ideal| / RMS(ideal)
  (nothing taken off) are printed beside them for every value.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O

NORM_TOL = 1e-2
STAT_RTOL = 1e-5
ROW_ALIGN = 128


def np64(t):
    if t is None:
        return None
    if not hasattr(t, "detach"):
        return np.asarray(t, dtype=np.float64)
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy().astype(np.float64)


def half_ulp_bf16(v):
    """Half a bfloat16 ulp of each value (0 for 0): the largest error one
    round-to-nearest into bf16 can make.  bf16 keeps 8 significant bits, so a
    value in [2^e, 2^(e+1)) has ulp 2^(e-7)."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    out = np.zeros_like(v)
    nz = v > 0
    out[nz] = np.exp2(np.floor(np.log2(v[nz])) - 8.0)
    return out


def norm_err(gpu, ref, output_rounding=False) -> float:
    """max_i (|gpu_i - ref_i| - a_i)+ / RMS(ref), a_i = half a bf16 ulp of
    gpu_i when ``output_rounding`` (the GPU stored the value in bf16), else 0."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = np.abs(gpu - ref)
    if output_rounding:
        diff = np.maximum(diff - half_ulp_bf16(gpu), 0.0)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    if rms == 0.0:
        return float(diff.max()) if diff.size else 0.0
    return float(diff.max()) / rms


def bf16_round(a):
    """Round-to-nearest-even to bfloat16, back in float64 (storage model)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(
        torch.bfloat16).double().numpy()


def frob_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = float(np.linalg.norm(ref))
    return float(np.linalg.norm(gpu - ref)) / n if n else float(np.linalg.norm(gpu))


def bf16_neighbours(v):
    """The two bf16 values bracketing each fp64 value (equal when v is one)."""
    v = np.asarray(v, dtype=np.float64)
    r = bf16_round(v)
    a = np.abs(r)
    ulp = np.where(a > 0, np.exp2(np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7), 2.0 ** -133)
    # the neighbour on the other side of v (one ulp of r away; at a power of
    # two below r the spacing halves, which the +-ulp/2 test below covers)
    other = np.where(v >= r, r + ulp, r - ulp)
    other_half = np.where(v >= r, r + ulp / 2, r - ulp / 2)
    return r, other, other_half


def fp16_neighbours(v):
    """As bf16_neighbours for IEEE binary16 (the MX training step's a, b):
    the rounding of v, the neighbour on the other side of v, and the same
    neighbour again (numpy's float16 steps across binade edges exactly)."""
    v = np.asarray(v, dtype=np.float64)
    r16 = np.clip(v, -65504.0, 65504.0).astype(np.float16)
    r = r16.astype(np.float64)
    up = np.nextafter(r16, np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(r16, np.float16(-np.inf)).astype(np.float64)
    other = np.where(v >= r, up, dn)
    return r, other, other


class AdoptStored:
    """Storage hook for the oracle (``rnd=``) that continues from the GPU's
    own stored bf16 values wherever they are a valid rounding.

    The layer keeps h, each routed slot's output (out), a, b, d_out, da, db
    and each routed slot's dx contribution (dxe) in bf16, each the rounding of
    an fp32 result (the MX training step keeps a and b in fp16: points a16,
    b16).  Where that result lies within its accumulation error of
    a rounding boundary, either bf16 neighbour is a correct outcome, as a
    near-tie in routing may go either way; one such flip in a heavy-tailed
    weight gradient moves it by a bf16 ulp of its largest product, which can
    exceed 1e-2 of the RMS on its own.  So, as for near-tie routing, each GPU
    stored value is checked to be a valid outcome -- the bf16 rounding of the
    oracle's value, the other bf16 neighbour of that value, or within
    2^-12 x RMS of its group where cancellation leaves the value tiny -- and
    the oracle then continues from it.  The outputs compared afterwards
    differ from the oracle only by the kernels' own arithmetic.  Every
    difference is counted: at most ``max_frac`` of the elements of any
    storage point may take the other neighbour, and none may be invalid.

    ``gpu``: point -> (routed, shared): arrays of rows [R][n] / [T][n], or
    functions of row indices returning those rows (stored_from_layer).
    ``row_of_pair``: permuted row of pair t*k + j.
    """

    def __init__(self, gpu, row_of_pair, k, max_frac=1e-2, tokens=None):
        self.gpu = gpu
        self.row_of_pair = np.asarray(row_of_pair)
        self.k = k
        self.max_frac = max_frac
        self.tokens = None if tokens is None else np.asarray(tokens)   # oracle row -> token
        self.stats = {}

    def adopt(self, point, v, s):
        """Validate GPU values ``s`` against the oracle's unrounded ``v``;
        returns s."""
        v = np.asarray(v, dtype=np.float64)
        s = np.asarray(s, dtype=np.float64)
        r, other, other_half = (fp16_neighbours if point.endswith("16") else bf16_neighbours)(v)
        rms = float(np.sqrt(np.mean(v * v))) if v.size else 0.0
        ok = (s == r) | (s == other) | (s == other_half) | (np.abs(s - v) <= 2.0 ** -12 * rms)
        st = self.stats.setdefault(point, [0, 0, 0])
        st[0] += v.size
        st[1] += int((s != r).sum())
        st[2] += int((~ok).sum())
        return s

    def store(self, point, v, where):
        routed, shared = self.gpu[point]
        rows = np.asarray(where["rows"])
        if self.tokens is not None:
            rows = self.tokens[rows]
        src, idx = (shared, rows) if where.get("shared") else \
            (routed, self.row_of_pair[rows * self.k + where["j"]])
        s = src(idx) if callable(src) else src[idx]
        return self.adopt(point, v, s)

    def __call__(self, v):
        return bf16_round(v)

    def quantised(self, point, v, q, where):
        """An MXFP8 quantisation point of a routed expert (q_h, q_d_out,
        q_d_gu; the oracle's mx_oracle._quantised): the GPU's codes and block
        scales for these rows, each checked to be the quantisation of some
        value within the kernels' fp32 error of the oracle's unquantised v
        (mx_valid), and continued from; q is the oracle's own Q(v).  At most
        max_frac_q of the codes may differ from the oracle's, none may be
        invalid.  Points without a GPU source return q."""
        from oracle import mx_oracle as M
        if point not in self.gpu:
            return q
        rows = np.asarray(where["rows"])
        if self.tokens is not None:
            rows = self.tokens[rows]
        codes, sbytes = self.gpu[point][0](self.row_of_pair[rows * self.k + where["j"]])
        valid, other = mx_valid(v, codes, sbytes)
        st = self.stats.setdefault(point, [0, 0, 0])
        st[0] += codes.size
        st[1] += int(other.sum())
        st[2] += int((~valid).sum())
        return M.mx_dequantize(codes, sbytes)

    def check(self, chk):
        """Rows for a Checker: invalid choices (must be 0) and the fraction
        of elements that took the other neighbour (<= max_frac; for the MX
        quantisation points, <= max_frac_q of the codes)."""
        for p, (n, diff, bad) in sorted(self.stats.items()):
            q = p.startswith("q_")
            chk.rows.append((f"{'quantised' if q else 'stored'} {p}: invalid", float(bad), 0.0))
            chk.rows.append((f"{'quantised' if q else 'stored'} {p}: other "
                             f"{'code' if q else 'rounding'} (frac)", diff / max(n, 1),
                             MAX_FRAC_Q if q else self.max_frac))


# at most this fraction of a quantisation point's codes may differ from the
# oracle's (each a valid quantisation of a value within fp32 error)
MAX_FRAC_Q = 1e-3


def mx_valid(v, codes, sbytes, tol_rel=2.0 ** -18, tol_abs=2.0 ** -16):
    """Is each GPU MX code [n][K] (with its block scale bytes [n][K/32]) the
    quantisation of a value within e = tol_rel |v| + tol_abs amax(block) of
    the oracle's v?  The block scale must be the one of v's block maximum,
    or one off where that maximum lies within the tolerance of a power of
    two; each code must lie between the e4m3 roundings, under the GPU's
    scale, of v - e and v + e (the rounding is monotone).  The tolerances
    cover fp32 against fp64 arithmetic (products, dot products over a few
    thousand terms) and are far below an e4m3 step (2^-4 relative).
    Returns (valid, differs from the oracle's own code or scale), each
    [n][K] bool."""
    from oracle import mx_oracle as M
    v = np.asarray(v, dtype=np.float64)
    n, K = v.shape
    b = v.reshape(n, K // 32, 32)
    amax = np.abs(b).max(axis=-1)
    c_o, s_o = M.mx_quantize(v)
    sg = np.asarray(sbytes).astype(np.int64)
    so = s_o.astype(np.int64)
    t = tol_rel + tol_abs
    crosses = M.mx_scale_exp(amax * (1 + t)) != M.mx_scale_exp(amax * (1 - t))
    scale_ok = (sg == so) | ((np.abs(sg - so) == 1) & crosses)
    e = tol_rel * np.abs(b) + tol_abs * amax[..., None]
    sc = np.exp2(sg - 127.0)[..., None]
    lo = M.e4m3_decode(M.e4m3_round((b - e) / sc))
    hi = M.e4m3_decode(M.e4m3_round((b + e) / sc))
    g = M.e4m3_decode(np.asarray(codes).reshape(n, K // 32, 32))
    ok = (g >= lo) & (g <= hi) & scale_ok[..., None]
    other = (np.asarray(codes) != c_o).reshape(n, K // 32, 32) | (sg != so)[..., None]
    return ok.reshape(n, K), other.reshape(n, K)


def mx_rows_from(q_buf, s_buf, R, K):
    """Function of permuted rows -> (codes [n][K], scale bytes [n][K/32]) of
    an MX buffer pair: codes [R][K] and scale atoms [R/128][K/128][512]
    (row r, block kb at byte (r%32)*16 + ((r/32)%4)*4 + kb%4 of its atom)."""
    import torch
    cache = {}

    def get(rows):
        rows = np.asarray(rows, dtype=np.int64)
        if "s" not in cache:
            cache["s"] = s_buf.cpu().numpy()
        q = q_buf[:R * K].view(R, K)[torch.as_tensor(rows, device=q_buf.device)]
        r = rows[:, None]
        kb = np.arange(K // 32)[None, :]
        idx = ((r >> 7) * (K // 128) + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3)
        return q.cpu().numpy(), cache["s"][idx]
    return get


def stored_from_layer(lay, with_backward, cols=None, shared_cols=None):
    """The GPU's stored bf16 values by storage point: point -> (routed, shared),
    each a function of row indices returning fp64 rows (shared is None
    without a shared expert).  Only the rows asked for are copied from the
    device.  ``cols`` / ``shared_cols`` restrict the hidden units (columns of
    h, a, b, da, db) to a subset, in that order."""
    import torch
    b = lay.bufs
    H = lay.cfg.H
    Hs = lay.cfg.n_shared * lay.cfg.H_shared

    def pick(t, c0, n, sub):
        if t is None:
            return None
        sel = None if sub is None else torch.as_tensor(np.asarray(sub) + c0, device=t.device)

        def get(rows):
            r = t[torch.as_tensor(np.asarray(rows, dtype=np.int64), device=t.device)]
            r = r[:, c0:c0 + n] if sel is None else r[:, sel]
            return np64(r)
        return get
    out = {"h": (pick(b["h"], 0, H, cols), pick(b.get("s_h"), 0, Hs, shared_cols)),
           # each routed slot's expert output (the shared expert's is not kept)
           "out": (pick(b["out_perm"], 0, lay.cfg.d, None), None)}
    if b.get("ab") is not None:
        out["a"] = (pick(b["ab"], 0, H, cols), pick(b.get("s_ab"), 0, Hs, shared_cols))
        out["b"] = (pick(b["ab"], H, H, cols), pick(b.get("s_ab"), Hs, Hs, shared_cols))
    if with_backward:
        it = lay.intermediates()
        out["d_out"] = (pick(it["d_out"], 0, lay.cfg.d, None), None)
        out["da"] = (pick(it["d_gu"], 0, H, cols), pick(it.get("ds_gu"), 0, Hs, shared_cols))
        out["db"] = (pick(it["d_gu"], H, H, cols), pick(it.get("ds_gu"), Hs, Hs, shared_cols))
        out["dxe"] = (pick(it["dx_perm"], 0, lay.cfg.d, None), None)
    mx = getattr(lay, "mx", None)
    if mx is not None:
        # the MXFP8 path's quantised operands (codes + block scales per row;
        # those of h and d_gu only for whole rows of hidden units)
        R = lay.R_cap
        if mx.get("ab16") is not None:
            import torch
            ab16 = mx["ab16"].view(torch.float16)[:R * 2 * H].view(R, 2 * H)
            out["a16"] = (pick(ab16, 0, H, cols), None)
            out["b16"] = (pick(ab16, H, H, cols), None)
        if cols is None:
            out["q_h"] = (mx_rows_from(mx["h_q"], mx["h_s"], R, H), None)
        if with_backward and mx.get("dout_q") is not None:
            out["q_d_out"] = (mx_rows_from(mx["dout_q"], mx["dout_s"], R, lay.cfg.d), None)
            if cols is None:
                out["q_d_gu"] = (mx_rows_from(mx["dgu_q"], mx["dgu_s"], R, 2 * H), None)
    return out


def _is_bf16(t):
    return hasattr(t, "dtype") and t.dtype == torch.bfloat16


class Checker:
    """Collects every comparison of a test, then fails with the full table.

    close(name, gpu, ref, tol): max normalised |gpu - ref| <= tol, for values
        compared directly (fp32 logits, identities such as dW_r = x^T dL).
    layer(name, gpu, exact, ideal, tol): the bound for bf16 outputs and
        gradients (module docstring): max normalised |gpu - ideal| <= tol,
        with half a bf16 ulp of a bf16-stored GPU value taken off each
        difference, and Frobenius-relative |gpu - exact| <= tol.  The plain
        max normalised errors against both are recorded without a bound.
    """

    def __init__(self):
        self.rows = []

    def close(self, name, gpu, ref, tol=NORM_TOL):
        e = norm_err(np64(gpu), ref, _is_bf16(gpu))
        self.rows.append((name, e, tol))
        return e

    def layer(self, name, gpu, exact, ideal, tol=NORM_TOL):
        g = np64(gpu)
        e = norm_err(g, ideal, _is_bf16(gpu))
        self.rows.append((name + "|gpu-ideal|max", e, tol))
        self.rows.append((name + "|gpu-exact|F", frob_err(g, exact), tol))
        self.rows.append((name + "|gpu-exact|max,plain", norm_err(g, exact), float("inf")))
        self.rows.append((name + "|gpu-ideal|max,plain", norm_err(g, ideal), float("inf")))
        return e

    def done(self):
        bad = [r for r in self.rows if not (r[1] <= r[2])]
        table = ", ".join(f"{n}={e:.2e}" for n, e, _ in self.rows)
        print("errors:", table)
        assert not bad, "over tolerance: " + ", ".join(f"{n} {e:.3e} > {t:.2e}"
                                                       for n, e, t in bad) + f" | all: {table}"


def assert_route_matches(bufs, ref):
    """The GPU's routing outputs against the oracle's route run on the same
    fp32 logits: selection and counts bit for bit, gates, f, p, aux and the
    routing metrics within STAT_RTOL."""
    import pytest
    b = bufs
    np.testing.assert_array_equal(b["topk_idx"].cpu().numpy(), ref["topk_idx"])
    np.testing.assert_array_equal(b["counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_allclose(np64(b["gates"]), ref["gates"], rtol=STAT_RTOL, atol=1e-7)
    np.testing.assert_allclose(np64(b["f"]), ref["f"], rtol=STAT_RTOL, atol=0)
    np.testing.assert_allclose(np64(b["p"]), ref["p"], rtol=STAT_RTOL, atol=1e-9)
    assert float(b["aux"][0]) == pytest.approx(ref["aux"], rel=STAT_RTOL)
    if b.get("router_stats") is not None:
        st = b["router_stats"].cpu().numpy().astype(np.float64)
        assert st[0] == pytest.approx(ref["z_loss"], rel=STAT_RTOL)
        assert st[1] == pytest.approx(ref["entropy"], rel=STAT_RTOL, abs=1e-7)
        assert (st[2], st[3], st[5], st[6]) == (ref["count_min"], ref["count_max"],
                                                ref["unused"], ref["T_real"])
        assert st[4] == pytest.approx(ref["count_cv"], rel=1e-6, abs=1e-7)


def route_on_gpu_logits(bufs, inp, k, norm_topk):
    """The oracle's route on the fp32 logits the GPU computed (so that the
    selection sees the same keys), with the inputs' bias and PAD mask."""
    bias = inp.get("bias")
    valid = inp.get("valid")
    return O.route(bufs["logits"].cpu().numpy(), k,
                   bias=None if bias is None else bias.cpu().numpy(),
                   valid=None if valid is None else valid.cpu().numpy(),
                   norm_topk=bool(norm_topk))


def assert_close(name, gpu, ref, tol=NORM_TOL):
    c = Checker()
    c.close(name, gpu, ref, tol)
    c.done()


def padded_layout(topk_idx, E):
    """Row of every (t, j) pair in the padded expert-contiguous layout.

    The order within the rows is the oracle's stable counting sort; each
    expert segment then starts at the next multiple of 128 rows (the layout
    the library documents).  Returns (offsets, row_offsets, row_of_pair,
    perm_padded) with -1 for PAD pairs / pad rows.
    """
    offsets, perm, inv = O.permute(topk_idx, E)
    counts = np.diff(offsets)
    padded = (counts + ROW_ALIGN - 1) // ROW_ALIGN * ROW_ALIGN
    row_offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)
    row_of_pair = np.full(inv.shape[0], -1, dtype=np.int64)
    R = int(row_offsets[-1])
    perm_padded = np.full(R, -1, dtype=np.int64)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        rows = row_offsets[e] + np.arange(seg.shape[0])
        row_of_pair[seg] = rows
        perm_padded[rows] = seg
    return offsets, row_offsets, row_of_pair, perm_padded


def routing_margin(key, k):
    """Gap between the k-th and (k+1)-th largest key of each row (inf if k==E)."""
    key = np.asarray(key, dtype=np.float64)
    if k >= key.shape[1]:
        return np.full(key.shape[0], np.inf)
    s = -np.sort(-key, axis=1)
    return s[:, k - 1] - s[:, k]


def logit_error_bound(x, Wr):
    """A bound on |fp32 logits - exact| for any summation order:
    (2d + 2) * eps32 * sum_c |x_c W_ce|."""
    xa = np.abs(np.asarray(x, dtype=np.float64))
    wa = np.abs(np.asarray(Wr, dtype=np.float64))
    d = xa.shape[1]
    eps = 2.0 ** -24
    return (2 * d + 2) * eps * (xa @ wa)


def reconcile_selection(gpu_topk, key_exact, bound, k, real):
    """Selection to compare against, allowing only the freedom fp32 rounding
    gives.  For tokens whose k-th/(k+1)-th key gap exceeds twice the logit
    error bound the choice is unique and the GPU must match the oracle.  For
    the rest, the GPU's choice is accepted if it is a valid top-k within that
    bound.  Returns (selection, number of near-tie tokens adopted)."""
    key = np.asarray(key_exact, dtype=np.float64)
    T, E = key.shape
    ref_sel = O.select_topk(key, k)
    margin = routing_margin(key, k)
    # logit rounding on both sides, plus the fp32 rounding of (logit + bias)
    tol = 2.0 * bound.max(axis=1) + 2.0 ** -22 * np.abs(key).max(axis=1) + 1e-30
    gpu = np.asarray(gpu_topk)
    adopted = 0
    sel = ref_sel.copy()
    for t in range(T):
        if not real[t]:
            continue
        if np.array_equal(gpu[t], ref_sel[t]):
            continue
        assert margin[t] <= tol[t] or _slot_tie(key[t], ref_sel[t], tol[t]), \
            f"token {t}: selection differs with margin {margin[t]:.3e} > {tol[t]:.3e}"
        g = gpu[t]
        assert len(set(g.tolist())) == k and (g >= 0).all() and (g < E).all()
        others = np.setdiff1d(np.arange(E), g)
        kth = key[t, g].min()
        if others.size:
            assert kth >= key[t, others].max() - tol[t], f"token {t}: invalid near-tie choice"
        sk = key[t, g]
        assert (sk[:-1] >= sk[1:] - tol[t]).all(), f"token {t}: slot order invalid"
        sel[t] = g
        adopted += 1
    return sel, adopted


def _slot_tie(row_key, sel, tol):
    sk = row_key[sel]
    return bool((np.abs(np.diff(sk)) <= tol).any())
