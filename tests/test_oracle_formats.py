"""Pins of the oracle's number-format codecs against independent libraries
(ml_dtypes, torch float8/bfloat16 casts) and the OCP MX v1.0 tables stored
under tests/golden/."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_e2m1_table_golden():
    g = _golden("ocp_mx_format_tables.json")
    want = np.array(g["e2m1_values_by_code"], dtype=np.float64)
    got = F.e2m1_decode(np.arange(16, dtype=np.uint8))
    np.testing.assert_array_equal(got, want)


def test_e2m1_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(16, dtype=np.uint8)
    ref = codes.view(ml.float4_e2m1fn).astype(np.float64)
    np.testing.assert_array_equal(F.e2m1_decode(codes), ref)


def test_e4m3_decode_vs_torch_and_ml_dtypes():
    codes = np.arange(256, dtype=np.uint8)
    got = F.e4m3_decode(codes)
    ref_t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, ref_t)          # NaN positions compare equal
    ml = pytest.importorskip("ml_dtypes")
    ref_m = codes.view(ml.float8_e4m3fn).astype(np.float64)
    np.testing.assert_array_equal(got, ref_m)


def test_e4m3_golden_points():
    g = _golden("ocp_mx_format_tables.json")["e4m3"]
    for code, val in g["points"]:
        assert F.e4m3_decode(np.uint8(int(code, 16))) == val
    assert np.isnan(F.e4m3_decode(np.uint8(0x7F)))
    assert np.isnan(F.e4m3_decode(np.uint8(0xFF)))


def test_e8m0_vs_ml_dtypes():
    codes = np.arange(256, dtype=np.uint8)
    got = F.e8m0_decode(codes)
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127
    ml = pytest.importorskip("ml_dtypes")
    ref = codes.view(ml.float8_e8m0fnu).astype(np.float64)
    np.testing.assert_array_equal(got, ref)


def _random_f32(n, seed):
    rng = np.random.default_rng(seed)
    mag = np.ldexp(rng.uniform(1, 2, n), rng.integers(-14, 10, n))
    v = (mag * rng.choice([-1, 1], n)).astype(np.float32)
    return v


def _midpoints():
    """Every exact midpoint between adjacent finite E4M3 magnitudes (ties)."""
    vals = F.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    mids = mids.astype(np.float32)
    return np.concatenate([mids, -mids])


def test_e4m3_encode_vs_torch_cast():
    v = np.concatenate([_random_f32(200_000, 1), _midpoints(),
                        np.float32([0.0, -0.0, 1e-30, -1e-30, 448.0, 449.0, 463.9, 464.0,
                                    500.0, -1e6])])
    got = F.e4m3_encode(v)
    clamped = np.clip(v, -448.0, 448.0)
    ref = torch.from_numpy(clamped).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    v = np.concatenate([_random_f32(100_000, 2), _midpoints()])
    v = np.clip(v, -448.0, 448.0)
    ref = v.astype(ml.float8_e4m3fn).view(np.uint8)
    np.testing.assert_array_equal(F.e4m3_encode(v), ref)


def test_e4m3_encode_is_nearest_even_brute_force():
    """Brute force over all 254 finite codes: the encoder returns a nearest
    code, and on exact ties the one with an even mantissa."""
    vals = F.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = ~np.isnan(vals)
    v = np.concatenate([_random_f32(3000, 3), _midpoints()]).astype(np.float64)
    v = np.clip(v, -448, 448)
    for x in v:
        d = np.where(finite, np.abs(vals - x), np.inf)
        best = np.flatnonzero(d == d.min())
        code = int(F.e4m3_encode(np.float32(x)))
        if x == 0 or np.abs(x) < 2.0 ** -10:
            assert vals[code] == 0.0
            continue
        # among the nearest, prefer the same sign, then an even mantissa
        best = [b for b in best if np.sign(vals[b]) in (np.sign(x), 0)]
        if len(best) > 1:
            best = [b for b in best if (b & 1) == 0]
        assert code in best, (x, code, best)


def test_e4m3_roundtrip_every_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = F.e4m3_decode(codes)
    ok = ~np.isnan(vals)
    back = F.e4m3_encode(vals[ok].astype(np.float32))
    np.testing.assert_array_equal(back, codes[ok])


def test_bf16_round_vs_torch():
    v = np.concatenate([_random_f32(100_000, 4),
                        np.float32([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0])])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(F.bf16_round(v), ref)
    bits = F.f32_to_bf16_bits(v)
    np.testing.assert_array_equal(F.bf16_bits_to_f32(bits), ref)


def test_mxfp4_dequant_matches_ml_dtypes_layout():
    """Packed nibble order and the per-32 scale broadcast, against ml_dtypes'
    float4 decode of explicitly unpacked codes."""
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(5)
    packed = rng.integers(0, 256, (3, 64), dtype=np.uint8)        # K = 128
    scales = rng.integers(118, 136, (3, 4), dtype=np.uint8)
    lo = (packed & 0xF).view(np.uint8).view(ml.float4_e2m1fn).astype(np.float64)
    hi = (packed >> 4).view(np.uint8).view(ml.float4_e2m1fn).astype(np.float64)
    vals = np.empty((3, 128))
    vals[:, 0::2] = lo
    vals[:, 1::2] = hi
    sc = scales.view(ml.float8_e8m0fnu).astype(np.float64)
    want = vals * np.repeat(sc, 32, axis=1)
    np.testing.assert_array_equal(F.mxfp4_dequant(packed, scales), want)
