"""Planted mistakes in the oracle (on the CPU) must be caught by its pins.

Each test patches one oracle function with a plausible slip and reruns the
check of the pin that should catch it.
"""
import numpy as np
import pytest
import torch

import gen
from oracle import formats as F
from oracle import moe as M
from tests import test_oracle_pins as P


def test_swapped_nibbles_break_the_quantiser_bound(monkeypatch):
    good = F.q4_k_fields

    def swapped(blocks):
        d, dmin, sc, m, q = good(blocks)
        q2 = q.copy()
        q2[..., 0::2, :], q2[..., 1::2, :] = q[..., 1::2, :], q[..., 0::2, :]
        return d, dmin, sc, m, q2

    monkeypatch.setattr(F, "q4_k_fields", swapped)
    with pytest.raises(AssertionError):
        P.test_q4_k_dequant_within_quantiser_error_bound()


def test_swapped_scale_high_bits_break_the_bijection(monkeypatch):
    good = F.q4_k_fields

    def wrong(blocks):
        d, dmin, sc, m, q = good(blocks)
        s = np.asarray(blocks, dtype=np.uint8)[..., 4:16].astype(np.int64)
        sc = sc.copy()
        for j in range(4, 8):
            sc[..., j] = (s[..., j + 4] & 0x0F) | ((s[..., j] >> 6) << 4)   # min's top bits
        return d, dmin, sc, m, q

    monkeypatch.setattr(F, "q4_k_fields", wrong)
    with pytest.raises(AssertionError):
        P.test_q4_k_scale_fields_are_a_bijection()


def test_round_half_even_breaks_the_q8_1_worked_example(monkeypatch):
    monkeypatch.setattr(F, "_round_half_away", lambda v32: np.rint(v32.astype(np.float64)))
    with pytest.raises(AssertionError):
        P.test_q8_1_worked_example()


def test_s_from_sum_of_x_breaks_the_q8_1_worked_example(monkeypatch):
    good = F.q8_1_quantize

    def wrong(x):
        a = good(x)
        xb = np.asarray(x, np.float32).reshape(-1, 32).astype(np.float64)
        a["s"] = F.fp16(xb.sum(1))
        return a

    monkeypatch.setattr(F, "q8_1_quantize", wrong)
    with pytest.raises(AssertionError):
        P.test_q8_1_worked_example()


def test_ties_to_higher_index_break_the_hand_example(monkeypatch):
    monkeypatch.setattr(M, "topk_sort", lambda l, k=8: sorted(
        range(len(l)), key=lambda e: (-float(l[e]), -e))[:k])
    with pytest.raises(AssertionError):
        P.test_topk_hand_example()


def test_gate_up_swapped_breaks_the_tiny_literal(monkeypatch):
    good = M.matvec_bf16

    def ffn(fmt, gate, up, down, x, x_q8_1=None):
        g = good(up, x)
        u = good(gate, x)
        h = M.silu(g) * u
        return {"g": g, "u": u, "h": h, "y": good(down, h)}

    monkeypatch.setattr(M, "expert_ffn", ffn)
    with pytest.raises(AssertionError):
        P.test_expert_ffn_tiny_literal()


def test_unnormalised_weights_break_the_convex_combination(monkeypatch):
    monkeypatch.setattr(M, "softmax_selected",
                        lambda l, ids: np.exp(np.asarray(l, np.float64)[list(ids)]))
    with pytest.raises(AssertionError):
        P.test_routed_combination_is_convex_over_identical_experts()


def test_min_term_sign_flip_breaks_the_dequantised_product(monkeypatch):
    good = F.q4_k_fields

    def neg_min(blocks):
        d, dmin, sc, m, q = good(blocks)
        return d, -dmin, sc, m, q

    def wrong_matvec(w_rows, a):
        d, dmin, sc, m, _ = neg_min(F.q4_k_rows(w_rows))
        rows, nsb = d.shape
        isum = M.q4_k_block_dots(w_rows, a).reshape(rows, nsb, 8).astype(np.float64)
        da, sa = a["d"].reshape(nsb, 8), a["s"].reshape(nsb, 8)
        return (d[..., None] * sc * da[None] * isum - dmin[..., None] * m * sa[None]).reshape(rows, -1).sum(1)

    monkeypatch.setattr(M, "matvec_q4_k", wrong_matvec)
    with pytest.raises(AssertionError):
        P.test_q4_k_matvec_equals_dequantised_product_when_s_is_exact()


def test_missing_first_rounding_breaks_fused_equals_unfused(monkeypatch):
    def fused_no_t_round(a, b, c, w, eps):
        s = F.bf16(np.asarray(a) + np.asarray(b) + np.asarray(c))
        r = 1.0 / np.sqrt(np.mean(s * s) + eps)
        return s, F.bf16(s * r * np.asarray(w))

    monkeypatch.setattr(M, "add_rmsnorm3", fused_no_t_round)
    with pytest.raises(AssertionError):
        P.test_add_rmsnorm3_equals_unfused_chain_bit_exact()


def test_h_rounded_to_bf16_breaks_the_fp16_mode_bound(monkeypatch):
    from tests import test_oracle_float_pins as FP

    def wrong(fmt, gate, up, down, x):
        G, U, D = (F.fp16(F.fp32(M.dequant_rows(fmt, m))) for m in (gate, up, down))
        x16 = F.fp16(np.asarray(x, dtype=np.float64))
        g, u = G @ x16, U @ x16
        h = M.silu(g) * u
        return {"g": g, "u": u, "h": h, "y": D @ F.bf16(h)}   # bf16 where fp16 is meant

    monkeypatch.setattr(M, "expert_ffn_fp16", wrong)
    with pytest.raises(AssertionError):
        FP.test_fp16_mode_is_the_float_mode_up_to_the_rounding_of_h()


def test_gate_and_up_swapped_break_the_float_mode_brute_force(monkeypatch):
    from tests import test_oracle_float_pins as FP

    def wrong(fmt, gate, up, down, x, down_fmt=None):
        G, U = (M.dequant_rows(fmt, m) for m in (up, gate))   # swapped
        D = M.dequant_rows(down_fmt or fmt, down)
        xx = np.asarray(x, dtype=np.float64)
        g, u = G @ xx, U @ xx
        h = M.silu(g) * u
        return {"g": g, "u": u, "h": h, "y": D @ h}

    monkeypatch.setattr(M, "expert_ffn_float", wrong)
    with pytest.raises(AssertionError):
        FP.test_float_mode_equals_integer_brute_force()


# ----------------------------------------------------------------------------
# Slips in the parity criteria: caught by tests/test_oracle_parity_pins.py
# ----------------------------------------------------------------------------

def test_ulp_exponent_off_by_one_breaks_the_spacing_pin(monkeypatch):
    from oracle import parity as PP
    from tests import test_oracle_parity_pins as PR

    def wrong(v):
        v = np.abs(np.asarray(v, dtype=np.float64))
        _, e = np.frexp(np.where(v > 0, v, 1.0))
        return np.where(v > 0, np.ldexp(1.0, np.maximum(e - 7, -133)), np.ldexp(1.0, -133))

    monkeypatch.setattr(PP, "ulp_bf16", wrong)
    with pytest.raises(AssertionError):
        PR.test_ulp_bf16_is_the_spacing_of_adjacent_bf16_values()


def test_ids_check_without_the_gap_rule_breaks_the_near_tie_pin(monkeypatch):
    from oracle import parity as PP
    from tests import test_oracle_parity_pins as PR
    good = PP.ids_valid
    monkeypatch.setattr(PP, "ids_valid", lambda g, r, l, tie_rel=PP.TIE_REL: good(g, r, l, 1.0))
    with pytest.raises(AssertionError):
        PR.test_ids_valid_near_tie_rule()


def test_parity_without_the_l2_bound_breaks_its_pin(monkeypatch):
    from oracle import parity as PP
    from tests import test_oracle_parity_pins as PR
    good = PP.float_parity
    monkeypatch.setattr(PP, "float_parity",
                        lambda g, o, rel_l2=PP.REL_L2, ulps=PP.ULPS: good(g, o, 1.0, ulps))
    with pytest.raises(AssertionError):
        PR.test_float_parity_relative_l2_boundary()


# ----------------------------------------------------------------------------
# Slips in the whole layer: caught by tests/test_oracle_layer_pins.py
# ----------------------------------------------------------------------------

def _slipped_layer_forward(slip):
    """oracle.moe.layer_forward with one planted mistake."""
    def lf(L, x, residual=None, ids=None, mode="int"):
        spec = L["spec"]
        xx = M.as_f64(x)
        res = xx if (residual is None or slip == "residual_is_x") else M.as_f64(residual)
        logits = M.router_logits(xx, L["w_router"])
        if ids is None:
            ids = M.topk_sort(logits, spec.top_k)
        if slip == "order_reversed":
            ids = list(reversed(ids))
        if slip == "softmax_over_all":
            full = np.exp(logits - logits.max())
            w = full[list(ids)] / full.sum()
        else:
            w = M.softmax_selected(logits, ids)
        f = M.moe_ffn(L, xx, ids, w, mode)
        shared = f["shared"]
        if spec.shared_inter > 0 and slip in ("gate_on_input", "gate_from_residual"):
            z = M.as_f64(L["w_sg"]) @ (res if slip == "gate_from_residual" else xx)
            gs = M.sigmoid(float(z))
            inp = gs * xx if slip == "gate_on_input" else xx
            ys = M.expert_ffn("bf16", L["sh_gate"], L["sh_up"], L["sh_down"], inp)["y"]
            shared = ys if slip == "gate_on_input" else gs * ys
        routed16 = f["routed"] if slip == "routed_unrounded" else F.bf16(f["routed"])
        shared16 = F.bf16(shared)
        if spec.shared_inter > 0 and slip != "shared_dropped":
            s, y = M.add_rmsnorm3(routed16, shared16, res, M.as_f64(L["w_norm"]), spec.eps)
        else:
            s, y = M.add_rmsnorm2(routed16, res, M.as_f64(L["w_norm"]), spec.eps)
        return {"logits": logits, "ids": list(ids), "w": w, "routed": f["routed"],
                "routed_bf16": routed16, "shared": shared, "shared_bf16": shared16, "sum": s,
                "y": y}
    return lf


@pytest.mark.parametrize("slip", ["residual_is_x", "order_reversed", "softmax_over_all",
                                  "gate_on_input", "gate_from_residual", "routed_unrounded",
                                  "shared_dropped"])
def test_layer_slips_break_the_worked_example(monkeypatch, slip):
    from tests import test_oracle_layer_pins as LP
    monkeypatch.setattr(M, "layer_forward", _slipped_layer_forward(slip))
    with pytest.raises(AssertionError):
        LP.test_layer_worked_example()


def test_unslipped_copy_passes_the_worked_example(monkeypatch):
    """The copy used for the slips is faithful when no slip is planted."""
    from tests import test_oracle_layer_pins as LP
    monkeypatch.setattr(M, "layer_forward", _slipped_layer_forward(None))
    LP.test_layer_worked_example()
    LP.test_layer_worked_example_without_shared_expert()


def test_unrounded_routed_changes_the_folded_sum_itself():
    """The worked example's residual makes the bf16 rounding of routed before
    the fold visible in `sum`, not only in the stored routed output."""
    from tests import test_oracle_layer_pins as LP
    x, r = LP.hand_inputs()
    for with_shared in (True, False):
        good = M.layer_forward(LP.hand_layer(with_shared), x, r)
        bad = _slipped_layer_forward("routed_unrounded")(LP.hand_layer(with_shared), x, r)
        assert not np.array_equal(good["sum"], bad["sum"]), with_shared
