"""Helpers shared by the GPU parity tests: running the C-ABI layer on seeded
inputs and comparing it with the CPU oracle.

Tolerances: routing indices, counts, offsets and the permutation are
compared bit for bit; bf16 outputs and gradients by the maximum normalised
error  max|gpu - oracle| / RMS(oracle) <= 1e-2;  fp32 statistics (f, p, aux)
by relative error <= 1e-5.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O

NORM_TOL = 1e-2
STAT_RTOL = 1e-5
ROW_ALIGN = 128


BF16_U = 2.0 ** -8     # unit roundoff of bfloat16 (8 significant bits)


def np64(t):
    if t is None:
        return None
    if not hasattr(t, "detach"):
        return np.asarray(t, dtype=np.float64)
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy().astype(np.float64)


def norm_err(gpu, ref, rounding=0.0) -> float:
    """max_i (|gpu_i - ref_i| - rounding |gpu_i|)+ / RMS(ref).

    ``rounding`` is the unit roundoff of the format the GPU stored the value
    in (bf16: 2^-8): a value rounded once to that format lies within
    rounding * |stored| of the unrounded result, so that much of the
    difference is the output format, not the computation."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = np.abs(gpu - ref)
    if rounding:
        diff = np.maximum(diff - rounding * np.abs(gpu), 0.0)
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


class Checker:
    """Collects every comparison of a test, then fails with the full table.

    close(name, gpu, exact): max normalised error vs the exact oracle <= tol
        (the stated tolerance, literally; used for the layer output y).
    close2(name, gpu, exact, ideal): for values that pass through bf16
        storage between matrix products.  ``ideal`` is the oracle with bf16
        rounding at the layer's storage points and exact arithmetic
        otherwise, so |ideal - exact| is the error the storage format alone
        makes.  Requires
          max normalised |gpu - exact| <= 2 * max normalised |ideal - exact| + tol
          Frobenius-relative |gpu - exact| <= tol.
    """

    def __init__(self):
        self.rows = []

    def close(self, name, gpu, ref, tol=NORM_TOL):
        rounding = BF16_U if (hasattr(gpu, "dtype") and gpu.dtype == torch.bfloat16) else 0.0
        e = norm_err(np64(gpu), ref, rounding)
        self.rows.append((name, e, tol))
        return e

    def close2(self, name, gpu, exact, ideal, tol=NORM_TOL):
        rounding = BF16_U if (hasattr(gpu, "dtype") and gpu.dtype == torch.bfloat16) else 0.0
        g = np64(gpu)
        storage = norm_err(ideal, exact)
        self.rows.append((name + "(max)", norm_err(g, exact, rounding), 2 * storage + tol))
        self.rows.append((name + "(F)", frob_err(g, exact), tol))
        self.rows.append((name + "[storage]", storage, float("inf")))

    def done(self):
        bad = [r for r in self.rows if not (r[1] <= r[2])]
        table = ", ".join(f"{n}={e:.2e}" for n, e, _ in self.rows)
        print("errors:", table)
        assert not bad, "over tolerance: " + ", ".join(f"{n} {e:.3e} > {t:.2e}"
                                                       for n, e, t in bad) + f" | all: {table}"


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
