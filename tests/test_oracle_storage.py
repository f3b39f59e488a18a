"""Pins of the oracle's storage-rounding hook (CPU only).

The GPU tests compare the layer with the oracle run with bf16 rounding at the
layer's storage points (``rnd=``): the hidden h, each routed slot's expert
output (kept until the gated sum), d_out = g dY of the routed rows, the
saved pre-activations a and b, the results (da, db) of the SwiGLU chain rule,
and each routed slot's dx contribution (kept until the slots are summed).
Those tolerances are only as good as the hook, so it is pinned here on a
one-token layer small enough to work out by hand.

The hook is given a coarse rounding that also records every value it is
handed: to the nearest multiple of 1/8, and of 1/12 for the two per-slot
values (out, dxe), whose values here would sit on a tie of the 1/8 grid.
The test checks
* that exactly the storage values are rounded, no more and no fewer (h, out,
  d_out, a, b, da, db, dxe for the routed expert; h, a, b, da, db for the
  shared expert, whose d_out is the input dY itself and whose output and dx
  are not kept per slot), and
* every output of the forward and backward against numbers written out below
  step by step.
The inputs were chosen so that each plausible misplacement of a rounding
(dropping one, rounding dH before the chain rule, rounding the shared
expert's dY, rounding the expert output) changes at least one of those
numbers; tests/test_oracle_mutations.py plants each of them.

Layer: T = 1, d = 1, E = 2 routed experts, k = 1 without renormalisation,
H = 1, one shared expert with H_s = 1, aux_coef = 0.  x = 1, W_r = [ln 3, 0],
so the logits are [ln 3, 0], the softmax is [3/4, 1/4], expert 0 is chosen
and its gate is g = 3/4.
"""
import math

import numpy as np

from oracle import moe_oracle as O


def q8(v):
    """Round to the nearest multiple of 1/8 (no ties occur below)."""
    return np.round(np.asarray(v, dtype=np.float64) * 8.0) / 8.0


def q12(v):
    """Round to the nearest multiple of 1/12 (no ties occur below)."""
    return np.round(np.asarray(v, dtype=np.float64) * 12.0) / 12.0


def qpoint(point, v):
    return q12(v) if point in ("out", "dxe") else q8(v)


class Spy:
    """A storage rounding (qpoint) that records the values it rounds.  Called
    as a plain function (which the oracle never does; a planted mistake may)
    it rounds to 1/8."""

    def __init__(self):
        self.seen = []

    def store(self, point, v, where):
        v = np.asarray(v, dtype=np.float64)
        self.seen.extend(v.reshape(-1).tolist())
        return qpoint(point, v)

    def __call__(self, v):
        v = np.asarray(v, dtype=np.float64)
        self.seen.extend(v.reshape(-1).tolist())
        return q8(v)


class NamedSpy:
    """The same rounding through the hook's store() form, recording which
    storage point and which rows each value belongs to."""

    def __init__(self):
        self.points = []

    def store(self, point, v, where):
        self.points.append((point, "shared" if where.get("shared") else
                            (where["e"], where["j"]), tuple(where["rows"].tolist())))
        return qpoint(point, v)


X = np.array([[1.0]])
WR = np.array([[math.log(3.0), 0.0]])
W_GU = np.array([[[1.3], [1.7]],          # expert 0: gate 1.3, up 1.7
                 [[0.5], [0.5]]])         # expert 1 (not chosen)
W_DOWN = np.array([[[1.1]], [[0.5]]])
WS_GU = np.array([[1.1], [2.2]])          # shared: gate 1.1, up 2.2
WS_DOWN = np.array([[0.35]])
DY = np.array([[-0.9]])
SIG = O.sigmoid

# ---- the routed expert, written out
A, B = 1.3, 1.7                            # a = x W_gate, b = x W_up
H_PRE = A * SIG(A) * B                     # silu(1.3) * 1.7 = 1.73670 ...
H = 1.75                                   # stored: nearest multiple of 1/8
OUT_PRE = H * 1.1                          # 1.925
OUT = 23 / 12                              # stored: nearest multiple of 1/12
G = 0.75
DOUT_PRE = G * -0.9                        # -0.675
DOUT = -0.625                              # stored
DH = DOUT * 1.1                            # -0.6875 (the dH product; not stored)
A_S, B_S = 1.25, 1.75                      # stored a, b
DA_PRE = DH * B_S * SIG(A_S) * (1 + A_S * (1 - SIG(A_S)))   # -1.19552 ...
DB_PRE = DH * A_S * SIG(A_S)                                 # -0.66799 ...
DA, DB = -1.25, -0.625                     # stored
DXE_PRE = DA * 1.3 + DB * 1.7              # -2.6875, the slot's dx contribution
DXE = -32 / 12                             # stored (1/12 grid)
# ---- the shared expert, written out (its d_out is dY itself)
AS, BS = 1.1, 2.2
HS_PRE = AS * SIG(AS) * BS                 # 1.81563 ...
HS = 1.875
DHS = -0.9 * 0.35                          # -0.315
AS_S, BS_S = 1.125, 2.25
DAS_PRE = DHS * BS_S * SIG(AS_S) * (1 + AS_S * (1 - SIG(AS_S)))   # -0.68257 ...
DBS_PRE = DHS * AS_S * SIG(AS_S)                                   # -0.26752 ...
DAS, DBS = -0.625, -0.25
# ---- outputs
Y = G * OUT + HS * 0.35                    # 1.4375 + 0.65625 = 2.09375
DG = -0.9 * OUT                            # -1.725 = <dY, out>
# raw gates: dL_e = s_e (u_e - sum_m s_m u_m), u = [dg, 0], s = [3/4, 1/4]
DL = np.array([0.75 * (DG - 0.75 * DG), 0.25 * (0.0 - 0.75 * DG)])
DW_DOWN = DOUT * H                         # -1.09375
DW_GU = np.array([DA, DB])                 # x = 1
DWS_DOWN = -0.9 * HS                       # -1.6875
DWS_GU = np.array([DAS, DBS])
DX = DXE + DAS * 1.1 + DBS * 2.2 + DL[0] * math.log(3.0)


def _forward():
    L = O.router_logits(X, WR)
    return O.forward(X, WR, W_GU, W_DOWN, WS_GU, WS_DOWN, k=1, norm_topk=False, logits=L)


def test_hand_case_routing():
    r = _forward()
    assert r["topk_idx"].tolist() == [[0]]
    np.testing.assert_allclose(r["gates"], [[0.75]], rtol=1e-15)


def test_forward_storage_points_by_hand():
    r = _forward()
    spy = Spy()
    y, routed = O.experts_forward(X, r["topk_idx"], r["gates"], W_GU, W_DOWN, WS_GU, WS_DOWN,
                                  rnd=spy)
    np.testing.assert_allclose(sorted(spy.seen), sorted([H_PRE, OUT_PRE, HS_PRE]), rtol=1e-14)
    np.testing.assert_allclose(routed[0, 0, 0], OUT, rtol=1e-14)
    np.testing.assert_allclose(y[0, 0], Y, rtol=1e-14)


def test_backward_storage_points_by_hand():
    r = _forward()
    spy = Spy()
    g = O.backward(X, WR, W_GU, W_DOWN, WS_GU, WS_DOWN, r, DY, norm_topk=False, aux_coef=0.0,
                   rnd=spy)
    # exactly the storage values are rounded: routed h, out, d_out, a, b, da,
    # db, dxe and shared h, a, b, da, db -- nothing else (dH, dY, outputs,
    # gradients)
    expect = [H_PRE, OUT_PRE, DOUT_PRE, A, B, DA_PRE, DB_PRE, DXE_PRE,
              HS_PRE, AS, BS, DAS_PRE, DBS_PRE]
    np.testing.assert_allclose(sorted(spy.seen), sorted(expect), rtol=1e-13)
    np.testing.assert_allclose(g["dg"], [[DG]], rtol=1e-14)
    np.testing.assert_allclose(g["d_logits"], [DL], rtol=1e-13)
    np.testing.assert_allclose(g["dW_down"][0], [[DW_DOWN]], rtol=1e-14)
    np.testing.assert_allclose(g["dW_gu"][0, :, 0], DW_GU, rtol=1e-14)
    assert not g["dW_gu"][1].any() and not g["dW_down"][1].any()
    np.testing.assert_allclose(g["dWs_down"], [[DWS_DOWN]], rtol=1e-14)
    np.testing.assert_allclose(g["dWs_gu"][:, 0], DWS_GU, rtol=1e-14)
    np.testing.assert_allclose(g["dx"], [[DX]], rtol=1e-13)
    np.testing.assert_allclose(g["dWr"], [DL], rtol=1e-13)


def test_stored_values_by_hand():
    """The written-out storage values themselves (the arithmetic above)."""
    assert q8(H_PRE) == H and q8(DOUT_PRE) == DOUT
    assert q12(OUT_PRE) == OUT and q12(DXE_PRE) == DXE
    assert (q8(A), q8(B)) == (A_S, B_S) and (q8(DA_PRE), q8(DB_PRE)) == (DA, DB)
    assert q8(HS_PRE) == HS and (q8(AS), q8(BS)) == (AS_S, BS_S)
    assert (q8(DAS_PRE), q8(DBS_PRE)) == (DAS, DBS)
    np.testing.assert_allclose([H_PRE, DA_PRE, DB_PRE], [1.7366953125, -1.1955222665,
                                                         -0.6679920682], rtol=1e-9)
    np.testing.assert_allclose([HS_PRE, DAS_PRE, DBS_PRE], [1.8156294555, -0.6825692215,
                                                            -0.2675229985], rtol=1e-9)
    assert abs(Y - 2.09375) < 1e-14


def test_storage_points_are_named_with_their_rows():
    """The store() form of the hook sees each storage point once per group
    of rows: routed expert 0, slot 0, token 0 -- h, out, d_out, a, b, da,
    db, dxe -- and the shared expert on token 0 -- h, a, b, da, db (no
    d_out: dY; no per-slot out or dxe)."""
    r = _forward()
    spy = NamedSpy()
    O.backward(X, WR, W_GU, W_DOWN, WS_GU, WS_DOWN, r, DY, norm_topk=False, aux_coef=0.0,
               rnd=spy)
    routed = sorted(p for p, w, rows in spy.points if w == (0, 0) and rows == (0,))
    shared = sorted(p for p, w, rows in spy.points if w == "shared" and rows == (0,))
    assert routed == sorted(["h", "out", "d_out", "a", "b", "da", "db", "dxe"])
    assert shared == sorted(["h", "a", "b", "da", "db"])
    assert len(spy.points) == 13
    spy = NamedSpy()
    O.experts_forward(X, r["topk_idx"], r["gates"], W_GU, W_DOWN, WS_GU, WS_DOWN, rnd=spy)
    assert sorted(map(repr, spy.points)) == sorted(map(repr, [("h", (0, 0), (0,)),
                                                              ("out", (0, 0), (0,)),
                                                              ("h", "shared", (0,))]))
