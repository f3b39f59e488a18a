"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (CPU only, through monkeypatch)
and checks that at least one pin from test_oracle_pins fails.  A pin set
that let any of these through would not be pinning the oracle.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O
import test_oracle_pins as P


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_reversed_tie_rule_is_caught(monkeypatch):
    def select_high_index_first(key, k):
        key = np.asarray(key)
        E = key.shape[1]
        order = np.argsort(-key[:, ::-1], axis=1, kind="stable")
        return (E - 1 - order)[:, :k]
    monkeypatch.setattr(O, "select_topk", select_high_index_first)
    assert _fails(P.test_selection_brute_force, 4, 2)
    assert _fails(P.test_equal_logits_tie_rule_and_balance)


def test_f_normalised_without_k_is_caught(monkeypatch):
    orig = O.route_stats

    def route_stats(s, idx, real, norm_topk=True):
        r = orig(s, idx, real, norm_topk)
        r["f"] = r["f"] * idx.shape[1]
        r["aux"] = s.shape[1] * float(np.dot(r["f"], r["p"]))
        return r
    monkeypatch.setattr(O, "route_stats", route_stats)
    assert _fails(P.test_equal_logits_tie_rule_and_balance)


def test_missing_renormalisation_is_caught(monkeypatch):
    orig = O.route_stats
    monkeypatch.setattr(O, "route_stats", lambda s, idx, real, norm_topk=True:
                        orig(s, idx, real, False))
    assert _fails(P.test_gates_renorm_and_raw)


def test_gate_and_up_swapped_is_caught(monkeypatch):
    def split_swapped(W_gu):
        H = W_gu.shape[-2] // 2
        return W_gu[..., H:, :], W_gu[..., :H, :]
    monkeypatch.setattr(O, "split_gu", split_swapped)
    assert _fails(P.test_dense_masked_brute_force)


def test_softmax_without_max_shift_is_caught(monkeypatch):
    def softmax_unshifted(L):
        with np.errstate(over="ignore", invalid="ignore"):
            z = np.exp(np.asarray(L, dtype=np.float64))
            return z / z.sum(axis=-1, keepdims=True)
    monkeypatch.setattr(O, "softmax", softmax_unshifted)
    assert _fails(P.test_softmax_closed_form)


def test_unstable_dispatch_order_is_caught(monkeypatch):
    def permute_tokens_descending(topk_idx, E):
        idx = np.asarray(topk_idx).reshape(-1)
        q_real = np.nonzero(idx >= 0)[0][::-1]
        perm = q_real[np.argsort(idx[q_real], kind="stable")]
        counts = np.bincount(idx[q_real], minlength=E)
        offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
        inv = np.full(idx.shape[0], -1, dtype=np.int64)
        inv[perm] = np.arange(perm.shape[0])
        return offsets, perm, inv
    monkeypatch.setattr(O, "permute", permute_tokens_descending)
    assert _fails(P.test_permute_invariants_and_brute_force)


def test_aux_gradient_sign_flip_is_caught(monkeypatch):
    orig = O.aux_logit_grad
    monkeypatch.setattr(O, "aux_logit_grad", lambda *a: -orig(*a))
    assert _fails(P.test_backward_matches_central_differences, True, True, False, 4, 0.0)


def test_dropped_silu_derivative_term_is_caught(monkeypatch):
    def swiglu_backward_wrong(dh, a, b):
        sa = O.sigmoid(a)
        return dh * b * sa, dh * O.silu(a)        # missing (1 + a (1 - s(a)))
    monkeypatch.setattr(O, "swiglu_backward", swiglu_backward_wrong)
    assert _fails(P.test_backward_matches_central_differences, True, True, False, 4, 0.0)


def test_router_input_gradient_dropped_is_caught(monkeypatch):
    orig = O.router_logit_grad
    monkeypatch.setattr(O, "router_logit_grad", lambda *a: 0.0 * orig(*a))
    assert _fails(P.test_backward_matches_central_differences, False, True, False, 4, 0.0)


def test_shared_expert_gated_is_caught(monkeypatch):
    orig = O.swiglu_parts
    calls = {"n": 0}

    def swiglu_half_shared(xr, Wg, Wu, Wd, rnd=None, where=None):
        out, a, b, h = orig(xr, Wg, Wu, Wd, rnd, where)
        # the shared expert is the call with the concatenated shared weights:
        # scale it as if it had a gate of 1/2
        if Wg.shape[0] == getattr(swiglu_half_shared, "Hs", -1):
            out = 0.5 * out
        return out, a, b, h
    swiglu_half_shared.Hs = 8                      # shared hidden of the pin's case
    monkeypatch.setattr(O, "swiglu_parts", swiglu_half_shared)
    assert _fails(P.test_k_equals_E_identical_experts_is_dense_ffn)


def test_z_loss_gradient_missing_factor_two_is_caught(monkeypatch):
    orig = O.z_logit_grad
    monkeypatch.setattr(O, "z_logit_grad", lambda L, real, z: orig(L, real, z / 2))
    assert _fails(P.test_backward_matches_central_differences, True, True, False, 4, 0.23)


# ---------------------------------------------------------------- MX oracle

import test_oracle_mx as PX
from oracle import mx_oracle as M


def test_mx_exponent_offset_7_is_caught(monkeypatch):
    orig = M.mx_scale_exp
    monkeypatch.setattr(M, "mx_scale_exp", lambda amax: np.minimum(orig(amax) + 1, 127))
    assert _fails(PX.test_mx_scale_closed_forms)
    assert _fails(PX.test_mx_quantize_is_nearest_on_the_block_grid)


def test_mx_ties_to_odd_is_caught(monkeypatch):
    tab = M.e4m3_table()

    def round_odd(q):
        q = np.asarray(q, dtype=np.float64)
        a = np.minimum(np.abs(q), M.E4M3_MAX)
        i = np.clip(np.searchsorted(tab, a, side="left"), 1, 126)
        d_lo, d_hi = a - tab[i - 1], tab[i] - a
        up = (d_hi < d_lo) | ((d_hi == d_lo) & (i % 2 == 1))
        code = np.where(up, i, i - 1)
        return (code | (np.signbit(q).astype(np.int64) << 7)).astype(np.uint8)
    monkeypatch.setattr(M, "e4m3_round", round_odd)
    assert _fails(PX.test_e4m3_round_matches_torch_float8)


def test_mx_blocks_along_wrong_axis_is_caught(monkeypatch):
    orig = M.mx_quantize

    def cols(v):
        v = np.asarray(v, dtype=np.float64)
        if v.ndim < 2 or v.shape[-2] % 32:
            return orig(v)
        c, s = orig(np.swapaxes(v, -1, -2))
        return np.swapaxes(c, -1, -2), s
    monkeypatch.setattr(M, "mx_quantize", cols)
    assert _fails(PX.test_mx_blocks_are_rows_of_32)


def test_mx_hidden_not_quantised_is_caught(monkeypatch):
    orig = O.experts_forward
    monkeypatch.setattr(O, "experts_forward",
                        lambda *a, rnd=None, **kw: orig(*a, **kw))
    assert _fails(PX.test_mx_experts_dense_masked_formulation)


def test_mx_shared_expert_left_unquantised_is_caught(monkeypatch):
    orig = M.experts_forward_mx

    def shared_exact(x, topk_idx, gates, W_gu, W_down, Ws_gu=None, Ws_down=None, valid=None):
        y, routed = orig(x, topk_idx, gates, W_gu, W_down, valid=valid)
        if Ws_gu is not None:
            sg, su = O.split_gu(np.asarray(Ws_gu, dtype=np.float64))
            shared, *_ = O.swiglu_parts(np.asarray(x, dtype=np.float64), sg, su,
                                        np.asarray(Ws_down, dtype=np.float64))
            y = y + shared
        return y, routed
    monkeypatch.setattr(M, "experts_forward_mx", shared_exact)
    assert _fails(PX.test_mx_experts_dense_masked_formulation)


# ---- the storage-rounding hook (tests/test_oracle_storage.py)

import inspect  # noqa: E402

import test_oracle_storage as S  # noqa: E402


def _storage_pins_fail():
    return (_fails(S.test_backward_storage_points_by_hand)
            or _fails(S.test_forward_storage_points_by_hand))


def _values_fail(monkeypatch):
    """The value checks alone (a spy that records nothing) also catch it."""
    class Quiet(S.Spy):
        def store(self, point, v, where):
            return S.qpoint(point, v)

        def __call__(self, v):
            return S.q8(v)
    monkeypatch.setattr(S, "Spy", Quiet)
    try:
        S.test_backward_storage_points_by_hand()
    except AssertionError:
        return True
    try:
        S.test_forward_storage_points_by_hand()
    except AssertionError:
        return True
    return False


def test_unrounded_hidden_is_caught(monkeypatch):
    orig = O.swiglu_parts
    monkeypatch.setattr(O, "swiglu_parts", lambda xr, Wg, Wu, Wd, rnd=None, where=None:
                        orig(xr, Wg, Wu, Wd, None, where))
    assert _storage_pins_fail()
    assert _values_fail(monkeypatch)


def test_rounded_shared_expert_output_is_caught(monkeypatch):
    """The shared expert's output is summed straight into y (no per-slot copy)."""
    orig = O.swiglu_parts

    def parts(xr, Wg, Wu, Wd, rnd=None, where=None):
        out, a, b, h = orig(xr, Wg, Wu, Wd, rnd, where)
        shared = where is not None and where.get("shared")
        return (rnd(out) if rnd and shared else out), a, b, h
    monkeypatch.setattr(O, "swiglu_parts", parts)
    assert _storage_pins_fail()
    assert _values_fail(monkeypatch)


@pytest.mark.parametrize("point", ["out", "dxe"])
def test_unrounded_per_slot_value_is_caught(monkeypatch, point):
    """A routed slot's expert output, or its dx contribution, not kept at its
    storage point before the slots are summed."""
    orig = O._store
    monkeypatch.setattr(O, "_store", lambda rnd, p, v, where: v if p == point
                        else orig(rnd, p, v, where))
    assert _storage_pins_fail()
    assert _values_fail(monkeypatch)


def test_unrounded_d_out_is_caught(monkeypatch):
    monkeypatch.setattr(O, "stored_d_out", lambda g, dY, rnd=None, where=None: g[:, None] * dY)
    assert _storage_pins_fail()
    assert _values_fail(monkeypatch)


def test_dh_rounded_before_the_chain_rule_is_caught(monkeypatch):
    orig = O.stored_swiglu_backward
    monkeypatch.setattr(O, "stored_swiglu_backward", lambda dh, a, b, rnd=None, where=None:
                        orig(rnd(dh) if rnd else dh, a, b, rnd, where))
    assert _storage_pins_fail()
    assert _values_fail(monkeypatch)


def test_dh_rounded_instead_of_da_db_is_caught(monkeypatch):
    def moved(dh, a, b, rnd=None, where=None):
        r = rnd or (lambda v: v)
        return O.swiglu_backward(r(dh), r(a), r(b))
    monkeypatch.setattr(O, "stored_swiglu_backward", moved)
    assert _storage_pins_fail()
    assert _values_fail(monkeypatch)


def test_unrounded_saved_preactivations_are_caught(monkeypatch):
    def exact_ab(dh, a, b, rnd=None, where=None):
        r = rnd or (lambda v: v)
        da, db = O.swiglu_backward(dh, a, b)
        return r(da), r(db)
    monkeypatch.setattr(O, "stored_swiglu_backward", exact_ab)
    assert _storage_pins_fail()
    assert _values_fail(monkeypatch)


def test_unrounded_da_db_are_caught(monkeypatch):
    def no_store(dh, a, b, rnd=None, where=None):
        r = rnd or (lambda v: v)
        return O.swiglu_backward(dh, r(a), r(b))
    monkeypatch.setattr(O, "stored_swiglu_backward", no_store)
    assert _storage_pins_fail()
    assert _values_fail(monkeypatch)


def test_rounded_shared_dY_is_caught(monkeypatch):
    src = inspect.getsource(O.shared_backward)
    needle = "stored_swiglu_backward(dY[rows] @ Ws_down_"
    assert needle in src
    ns = dict(vars(O))
    exec(src.replace(needle, "stored_swiglu_backward(rnd(dY[rows]) @ Ws_down_"), ns)
    monkeypatch.setattr(O, "shared_backward", ns["shared_backward"])
    assert _storage_pins_fail()
    assert _values_fail(monkeypatch)


# ---- the MXFP8 training step (tests/test_oracle_mx.py)

import test_oracle_mx as MXP  # noqa: E402
from oracle import mx_oracle as M  # noqa: E402


def test_mx_dgrad_weights_quantised_along_the_wrong_axis_are_caught(monkeypatch):
    monkeypatch.setattr(M, "roundtrip_k", lambda W, quant=None:
                        (quant or M.mx_roundtrip)(np.asarray(W, dtype=np.float64)))
    assert _fails(MXP.test_mx_backward_quantises_each_operand_along_its_reduction_axis)
    assert _fails(MXP.test_mx_backward_dense_masked_formulation)


def test_mx_dgrad_unquantised_d_gu_is_caught(monkeypatch):
    src = inspect.getsource(M.backward_mx)
    needle = '_quantised(rnd, "q_d_gu", d_gu, quant, where) @ qgu_k'
    assert needle in src
    ns = dict(vars(M))
    exec(src.replace(needle, "d_gu @ qgu_k"), ns)
    monkeypatch.setattr(M, "backward_mx", ns["backward_mx"])
    assert _fails(MXP.test_mx_backward_quantises_each_operand_along_its_reduction_axis)
    assert _fails(MXP.test_mx_backward_dense_masked_formulation)


@pytest.mark.parametrize("needle,planted", [
    ('dH = _quantised(rnd, "q_d_out", d_out_v,', 'dH = _quantised(rnd, "q_d_out", d_out,'),
    ('_store16(rnd, "a16", a, where)', 'mo._store(rnd, "a", a, where)'),
    ('_store16(rnd, "b16", b, where)', 'b'),
    ("d_gu = np.concatenate([da_v, db_v], axis=1)", "d_gu = np.concatenate([da, db], axis=1)"),
])
def test_mx_dgrad_quantising_the_bf16_copy_is_caught(monkeypatch, needle, planted):
    """Quantising the bf16-stored d_out or d_gu (a double rounding) instead
    of the values themselves; a in bf16 or b unrounded in the chain rule."""
    src = inspect.getsource(M.backward_mx)
    assert needle in src
    ns = dict(vars(M))
    exec(src.replace(needle, planted), ns)
    monkeypatch.setattr(M, "backward_mx", ns["backward_mx"])
    assert _fails(MXP.test_mx_backward_dense_masked_formulation)


def test_mx_training_shared_expert_in_mx_is_caught(monkeypatch):
    orig = M.experts_forward_mx
    monkeypatch.setattr(M, "experts_forward_mx", lambda *a, shared_mx=True, rnd=None, **k:
                        orig(*a, shared_mx=True, rnd=rnd, **k))
    assert _fails(MXP.test_mx_training_forward_has_the_bf16_shared_expert)
