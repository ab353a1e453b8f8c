"""Planted mistakes: each test breaks one step of the oracle (on the CPU,
through monkeypatch) and checks that at least one of the pins catches it.
This shows the pins are strong enough to detect a dropped term, a wrong
sign or index, or a swapped operand anywhere in the oracle."""
import numpy as np
import pytest

import sys, os
sys.path.insert(0, os.path.dirname(__file__))
import test_oracle_formats as TF  # noqa: E402
import test_oracle_forward as TW  # noqa: E402
import test_oracle_routing as TR  # noqa: E402
import test_oracle_split as TS  # noqa: E402
from oracle import formats as F
from oracle import moe as M


def _pins_forward():
    TW.test_exact_swiglu_golden_case()
    TW.test_forward_vs_brute_force(6, 3, 128, 64, 40, M.QUANT_W4A8)


def _expect_caught(pin):
    with pytest.raises(AssertionError):
        pin()


def test_pins_pass_unmutated():
    _pins_forward()
    TR.test_route_ties_lower_index_first()
    TR.test_expand_invariants_and_roundtrip()


def test_swapped_gate_up_is_caught(monkeypatch):
    def bad(g):
        I = g.shape[1] // 2
        return F.bf16_round((M.silu_f32(g[:, I:]) * g[:, :I]).astype(np.float32))
    monkeypatch.setattr(M, "swiglu_bf16", bad)
    _expect_caught(_pins_forward)


def test_dropped_token_scale_is_caught(monkeypatch):
    monkeypatch.setattr(M, "apply_row_scale", lambda acc, s: acc)
    _expect_caught(_pins_forward)


def test_wrong_nibble_order_is_caught(monkeypatch):
    def bad(packed):
        p = np.asarray(packed, dtype=np.uint8)
        out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
        out[..., 0::2] = p >> 4
        out[..., 1::2] = p & 0xF
        return out
    monkeypatch.setattr(F, "unpack_e2m1", bad)
    _expect_caught(_pins_forward)


def test_e8m0_bias_off_by_one_is_caught(monkeypatch):
    orig = F.e8m0_decode
    monkeypatch.setattr(F, "e8m0_decode", lambda c: orig(c) * 2.0)
    _expect_caught(TF.test_e8m0_vs_ml_dtypes)
    _expect_caught(_pins_forward)


def test_reversed_slot_weights_in_combine_is_caught(monkeypatch):
    orig = M.combine
    monkeypatch.setattr(M, "combine", lambda w, y, r: orig(w[:, ::-1].copy(), y, r))
    _expect_caught(lambda: TW.test_forward_vs_brute_force(6, 3, 128, 64, 40, M.QUANT_W4A8))


def test_tie_rule_reversed_is_caught(monkeypatch):
    orig = M.route

    def bad(logits, k):
        E = logits.shape[1]
        ids, w = orig(logits[:, ::-1].copy(), k)
        return (E - 1 - ids).astype(np.int32), w
    monkeypatch.setattr(M, "route", bad)
    _expect_caught(TR.test_route_ties_lower_index_first)


def test_round_half_up_encoder_is_caught(monkeypatch):
    orig = F.e4m3_encode

    def bad(v):
        v = np.asarray(v, dtype=np.float64)
        return orig(v * (1 + 2.0 ** -20))            # nudges ties upward
    monkeypatch.setattr(F, "e4m3_encode", bad)
    _expect_caught(TF.test_e4m3_encode_vs_torch_cast)


def test_unstable_expansion_is_caught(monkeypatch):
    orig = M.expand

    def bad(ids, w, E):
        rt = orig(ids, w, E)
        for e in range(E):               # reverse token order inside experts
            a, b = rt.offsets[e], rt.offsets[e + 1]
            rt.token_of_row[a:b] = rt.token_of_row[a:b][::-1].copy()
        return rt
    monkeypatch.setattr(M, "expand", bad)
    _expect_caught(TR.test_expand_invariants_and_roundtrip)


def test_transposed_gemm_operand_is_caught(monkeypatch):
    orig = M.Weights.dense

    def bad(self, which, e):
        d = orig(self, which, e)
        return d[::-1].copy()                # output features permuted
    monkeypatch.setattr(M.Weights, "dense", bad)
    _expect_caught(_pins_forward)


# ------------------------------------------------- W8A8 (MXFP8) and W4A16 modes
def _pins_forward_mx():
    TW.test_forward_vs_brute_force(6, 3, 128, 64, 40, M.QUANT_W8A8)


def _pins_forward_w16():
    TW.test_forward_vs_brute_force(6, 3, 128, 64, 40, M.QUANT_W4A16)


def test_mode_pins_pass_unmutated():
    _pins_forward_mx()
    _pins_forward_w16()
    TW.test_exact_golden_case_w8a8()
    TW.test_exact_golden_case_w4a16()


def test_mxfp8_round_up_instead_of_nearest_is_caught(monkeypatch):
    """E4M3 rounding of the MXFP8 quotient taken upward in magnitude: the
    golden case's h / X = 392 must give 384, not 416."""
    orig = F.e4m3_encode

    def bad(v):
        v = np.asarray(v, dtype=np.float64)
        codes = orig(v)
        dec = F.e4m3_decode(codes)
        up = np.abs(dec) < np.abs(v)                 # rounded down in magnitude
        bumped = np.where(up & ((codes & 0x7F) < 0x7E), codes + 1, codes)
        return bumped.astype(np.uint8)
    monkeypatch.setattr(F, "e4m3_encode", bad)
    _expect_caught(TW.test_exact_golden_case_w8a8)


def test_mxfp8_exponent_off_by_one_is_caught(monkeypatch):
    """X = 2^(floor(log2 amax) - 7) instead of - 8 (E4M3's emax is 8)."""
    orig = M.quantize_rows_mxfp8

    def bad(rows):
        _, sc = orig(rows)                                  # the correct exponents e
        v = np.asarray(rows, np.float32).astype(np.float64)
        blk = v.reshape(v.shape[:-1] + (v.shape[-1] // 32, 32))
        e1 = sc.astype(np.int32) - 127 + 1                  # one too large
        codes = F.e4m3_encode(blk / np.ldexp(1.0, e1)[..., None])
        return codes.reshape(v.shape).astype(np.uint8), (e1 + 127).astype(np.uint8)
    monkeypatch.setattr(M, "quantize_rows_mxfp8", bad)
    _expect_caught(_pins_forward_mx)
    _expect_caught(TW.test_exact_golden_case_w8a8)


def test_mxfp8_dropped_activation_scale_is_caught(monkeypatch):
    """The activation block scales dropped: codes of x / X paired with X = 1."""
    orig = M.quantize_rows_mxfp8

    def bad(rows):
        codes, sc = orig(rows)
        return codes, np.full_like(sc, 127)
    monkeypatch.setattr(M, "quantize_rows_mxfp8", bad)
    _expect_caught(_pins_forward_mx)
    _expect_caught(TW.test_exact_golden_case_w8a8)


def test_w4a16_h_not_rounded_to_bf16_is_caught(monkeypatch):
    """W4A16 feeds h to GEMM2 as bf16: skipping the rounding changes y."""
    def bad(g):
        I = g.shape[1] // 2
        return (M.silu_f32(g[:, :I]) * g[:, I:]).astype(np.float32) * np.float32(1.0 + 2.0 ** -7)
    monkeypatch.setattr(M, "swiglu_bf16", bad)
    _expect_caught(_pins_forward_w16)
    _expect_caught(TW.test_exact_golden_case_w4a16)


def _pin_route_and_quantize():
    for x, lg, k in TR._front_cases():
        TR.check_route_and_quantize(M.route_and_quantize, x, lg, k)


def test_route_and_quantize_pins_pass_unmutated():
    _pin_route_and_quantize()


@pytest.mark.parametrize("slip", ["bits_as_values", "negated_logits", "scale_reciprocal",
                                  "unstable_rows"])
def test_route_and_quantize_slips_are_caught(monkeypatch, slip):
    """Slips in the three steps route_and_quantize chains (the full-size GPU
    tests' bit-exact reference): quantising the raw bf16 bit patterns instead
    of their values, routing on negated logits, returning 448/amax as the
    scale, and an expansion that is not stable in token order."""
    orig_q, orig_route, orig_expand = M.quantize_rows_fp8, M.route, M.expand

    def bad(x_bits, logits, k):
        x = F.bf16_bits_to_f32(x_bits)
        if slip == "bits_as_values":
            x = np.asarray(x_bits, np.float32)
        lg = -np.asarray(logits, np.float32) if slip == "negated_logits" else logits
        ids, w = orig_route(np.asarray(lg, np.float32), k)
        rt = orig_expand(ids, w, logits.shape[1])
        if slip == "unstable_rows":
            for e in range(len(rt.counts)):
                a, b = rt.offsets[e], rt.offsets[e + 1]
                seg = slice(a, b)
                rt.token_of_row[seg] = rt.token_of_row[seg][::-1].copy()
        tq, ts = orig_q(x)
        if slip == "scale_reciprocal":
            ts = (np.float32(1.0) / ts).astype(np.float32)
        return rt, tq, ts
    _expect_caught(lambda: [TR.check_route_and_quantize(bad, x, lg, k)
                            for x, lg, k in TR._front_cases()])


def _split_variant(emax_off=7, residual=True, keep_lo=True):
    """A copy of the two-term split with one step changed."""
    def split(rows):
        v = np.asarray(rows, dtype=np.float32).astype(np.float64)
        shp = v.shape
        blk = v.reshape(shp[:-1] + (shp[-1] // 32, 32))

        def term(b):
            amax = np.abs(b).max(axis=-1)
            nz = amax > 0
            _, e2 = np.frexp(np.where(nz, amax, 1.0))
            e = np.where(nz, np.clip(e2 - 1 - emax_off, -127, 127), 0)
            sc = np.ldexp(1.0, e)[..., None]
            c = F.e4m3_encode(b / sc)
            return c, (e + 127).astype(np.uint8), F.e4m3_decode(c) * sc

        hc, hs, hv = term(blk)
        lc, ls, _ = term(blk - hv if residual else blk)
        if not keep_lo:
            lc = np.zeros_like(lc)
        return (np.concatenate([hc.reshape(shp), lc.reshape(shp)], -1).astype(np.uint8),
                np.concatenate([hs, ls], -1).astype(np.uint8))
    return split


def _pin_split():
    TS.test_split_hand_worked_block()
    TS.test_split_exact_over_every_bf16_value_of_14_binades()
    TS.test_split_error_bound_and_no_saturation()


@pytest.mark.parametrize("slip", [dict(emax_off=8), dict(emax_off=6), dict(residual=False),
                                  dict(keep_lo=False)],
                         ids=["ocp_emax", "one_binade_low", "lo_from_value", "dropped_lo"])
def test_split_slips_are_caught(monkeypatch, slip):
    _pin_split()
    monkeypatch.setattr(M, "split_rows_mxfp8x2", _split_variant(**slip))
    _expect_caught(_pin_split)
