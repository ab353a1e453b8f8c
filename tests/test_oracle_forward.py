"""Pins of the oracle's whole forward:
  * a closed-form golden case (tests/golden/exact_swiglu_case.json) whose
    intermediates and outputs are exact;
  * a brute-force formulation that runs every expert densely on every token
    and masks by routing (torch float64 + ml_dtypes decoding), independent of
    the oracle's grouped, expert-sorted formulation;
  * per-token independence (a token subset reproduces the full result)."""
import json
import os

import numpy as np
import pytest
import torch

import moe_inputs as MI
from oracle import formats as F
from oracle import moe as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
_VAL2CODE = {0: 0x0, 1: 0x2, -1: 0xA, 2: 0x4, -2: 0xC}


def _pack(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _exact_case_inputs(doc):
    E, H, I = doc["E"], doc["H"], doc["I"]
    rho, sigma, tau = (np.array(doc[k]) for k in ("rho", "sigma", "tau"))
    c1 = np.zeros((E, 2 * I, H), dtype=np.uint8)
    for e in range(E):
        for n in range(I):
            for p in doc["x_positions"]:
                c1[e, n, p] = _VAL2CODE[int(rho[e, n])]
                c1[e, I + n, p] = _VAL2CODE[int(sigma[e, n])]
    sf1 = np.full((E, 2 * I, H // 32), 127, dtype=np.uint8)
    sf1[:, :, 1] = doc["w1_block_scale_bytes"][1]
    c2 = np.vectorize(lambda v: _VAL2CODE[int(v)])(tau).astype(np.uint8)
    sf2 = np.full((E, H, I // 32), 127, dtype=np.uint8)
    x = np.zeros((2, H), dtype=np.float32)
    for t, p in enumerate(doc["x_positions"]):
        x[t, p] = 448.0
    xbits = F.f32_to_bf16_bits(x)
    W = M.Weights(_pack(c1), sf1, _pack(c2), sf2)
    return xbits, W


def test_exact_swiglu_golden_case():
    with open(os.path.join(GOLDEN, "exact_swiglu_case.json")) as f:
        doc = json.load(f)
    xbits, W = _exact_case_inputs(doc)
    I = doc["I"]
    rho, sigma = np.array(doc["rho"]), np.array(doc["sigma"])
    for case in doc["cases"]:
        k = case["top_k"]
        fw = M.forward(xbits, np.array(case["logits"], np.float32), W, k)
        np.testing.assert_array_equal(fw.out, np.array(case["expected_out"], np.float32))
        rt = fw.routing
        for r in range(len(rt.token_of_row)):
            t, e = rt.token_of_row[r], rt.expert_of_row[r]
            m = 1 if t == 0 else 2
            assert fw.x_scale[r] == 1.0
            assert fw.xq[r, doc["x_positions"][t]] == 0x7E
            np.testing.assert_array_equal(fw.g[r, :I], 448.0 * m * rho[e])
            np.testing.assert_array_equal(fw.g[r, I:], 448.0 * m * sigma[e])
            want_h = np.where(rho[e] > 0, (448.0 * m) ** 2 * sigma[e], 0.0)
            np.testing.assert_array_equal(fw.h[r], want_h)
            if np.any(rho[e] > 0):
                assert fw.h_scale[r] == 448.0 * m * m
                assert np.all((fw.hq[r][rho[e] > 0] & 0x7F) == 0x7E)
            else:
                assert fw.h_scale[r] == 1.0 and np.all(fw.hq[r] == 0)


_VAL2E4M3 = {0: 0x00, 1: 0x38, -1: 0xB8, 2: 0x40, -2: 0xC0}


def _exact_case_w8a8_weights(doc):
    """The golden case's weight values as MXFP8 (E4M3 codes, same scale bytes)."""
    E, H, I = doc["E"], doc["H"], doc["I"]
    rho, sigma, tau = (np.array(doc[k]) for k in ("rho", "sigma", "tau"))
    c1 = np.zeros((E, 2 * I, H), dtype=np.uint8)
    for e in range(E):
        for n in range(I):
            for p in doc["x_positions"]:
                c1[e, n, p] = _VAL2E4M3[int(rho[e, n])]
                c1[e, I + n, p] = _VAL2E4M3[int(sigma[e, n])]
    sf1 = np.full((E, 2 * I, H // 32), 127, dtype=np.uint8)
    sf1[:, :, 1] = doc["w1_block_scale_bytes"][1]
    c2 = np.vectorize(lambda v: _VAL2E4M3[int(v)])(tau).astype(np.uint8)
    sf2 = np.full((E, H, I // 32), 127, dtype=np.uint8)
    return M.Weights(c1, sf1, c2, sf2, mode=M.QUANT_W8A8)


def test_exact_golden_case_w4a16():
    """bf16 activations and bf16 h: the same exact outputs as W4A8."""
    with open(os.path.join(GOLDEN, "exact_swiglu_case.json")) as f:
        doc = json.load(f)
    xbits, W = _exact_case_inputs(doc)
    W = M.Weights(W.w1, W.w1_sf, W.w2, W.w2_sf, mode=M.QUANT_W4A16)
    I = doc["I"]
    rho, sigma = np.array(doc["rho"]), np.array(doc["sigma"])
    for case in doc["cases"]:
        fw = M.forward(xbits, np.array(case["logits"], np.float32), W, case["top_k"],
                       mode=M.QUANT_W4A16)
        np.testing.assert_array_equal(fw.out, np.array(case["expected_out_w4a16"], np.float32))
        assert fw.xq is None and fw.hq is None
        rt = fw.routing
        for r in range(len(rt.token_of_row)):
            t, e = rt.token_of_row[r], rt.expert_of_row[r]
            m = 1 if t == 0 else 2
            np.testing.assert_array_equal(fw.g[r, :I], 448.0 * m * rho[e])
            np.testing.assert_array_equal(fw.h[r], np.where(rho[e] > 0,
                                                            (448.0 * m) ** 2 * sigma[e], 0.0))


def test_exact_golden_case_w8a8():
    """MXFP8 blocks: x's block scale 1 with code 0x7E; h/X = +-392 rounds to
    +-384 (code 0x7C/0xFC) under the block scale 2^(9 + 2 log2 m)."""
    with open(os.path.join(GOLDEN, "exact_swiglu_case.json")) as f:
        doc = json.load(f)
    xbits, _ = _exact_case_inputs(doc)
    W = _exact_case_w8a8_weights(doc)
    I = doc["I"]
    rho = np.array(doc["rho"])
    mag, hbytes = doc["w8a8_h_code_magnitude"], doc["w8a8_h_scale_bytes"]
    for case in doc["cases"]:
        fw = M.forward(xbits, np.array(case["logits"], np.float32), W, case["top_k"],
                       mode=M.QUANT_W8A8)
        np.testing.assert_array_equal(fw.out, np.array(case["expected_out_w8a8"], np.float32))
        rt = fw.routing
        for r in range(len(rt.token_of_row)):
            t, e = rt.token_of_row[r], rt.expert_of_row[r]
            m = 1 if t == 0 else 2
            p = doc["x_positions"][t]
            assert fw.xq[r, p] == 0x7E and np.all(fw.x_scale[r] == 127)
            assert np.count_nonzero(fw.xq[r] & 0x7F) == 1
            np.testing.assert_array_equal(fw.g[r, :I], 448.0 * m * rho[e])
            if np.any(rho[e] > 0):
                assert fw.h_scale[r, 0] == hbytes[t]
                np.testing.assert_array_equal(fw.hq[r][rho[e] > 0] & 0x7F, mag)
                assert np.all(fw.hq[r][rho[e] < 0] & 0x7F == 0)
            else:
                assert fw.h_scale[r, 0] == 127 and np.all(fw.hq[r] & 0x7F == 0)


def _to_np(case):
    xbits = case.x.view(torch.int16).numpy().view(np.uint16)
    W = M.Weights(case.w1.numpy(), case.w1_sf.numpy(), case.w2.numpy(), case.w2_sf.numpy(),
                  mode=case.mode)
    return xbits, case.logits.numpy(), W


def brute_force(case, top_k, mode=MI.QUANT_W4A8):
    """Every expert on every token, dense, then masked: an independent
    formulation of the same forward (torch float64, ml_dtypes decoding), in
    each quantisation mode: W4A8 (per-token FP8), W8A8 (MXFP8 blocks, exponent
    from torch.frexp, codes from torch's E4M3 cast) and W4A16 (no activation
    quantisation)."""
    ml = pytest.importorskip("ml_dtypes")
    x = case.x.to(torch.float32)
    L = case.logits.to(torch.float64)
    T, E = L.shape
    idx = torch.arange(E)
    beats = (L[:, None, :] > L[:, :, None]) | ((L[:, None, :] == L[:, :, None])
                                               & (idx[None, None, :] < idx[None, :, None]))
    sel = beats.sum(-1) < top_k                          # fewer than k experts beat e
    p = torch.softmax(L, dim=1) * sel
    wsel = p / p.sum(1, keepdim=True)

    def quant(rows):
        amax = rows.abs().amax(1)
        nz = amax > 0
        s = torch.where(nz, amax / 448.0, torch.ones_like(amax))
        # tensor / tensor is IEEE division (a Python scalar divided by a
        # tensor is computed through a reciprocal and can differ by an ulp)
        inv = torch.where(nz, torch.full_like(amax, 448.0) / amax, torch.zeros_like(amax))
        q = (rows * inv[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn)
        return q.to(torch.float64), s

    def quant_mx(rows):
        blk = rows.to(torch.float64).reshape(rows.shape[0], -1, 32)
        amax = blk.abs().amax(-1)
        _, ex = torch.frexp(torch.where(amax > 0, amax, torch.ones_like(amax)))
        e = torch.where(amax > 0, (ex - 1 - 8).clamp(-127, 127), torch.zeros_like(ex))
        scale = torch.pow(2.0, e.to(torch.float64))[..., None]
        q = (blk / scale).clamp(-448, 448).to(torch.float8_e4m3fn).to(torch.float64)
        return (q * scale).reshape(rows.shape), torch.ones(rows.shape[0], dtype=torch.float64)

    def no_quant(rows):
        return rows.to(torch.float64), torch.ones(rows.shape[0], dtype=torch.float64)

    def dense(packed, sf):
        if mode == MI.QUANT_W8A8:
            v = packed.numpy().view(ml.float8_e4m3fn).astype(np.float64)
        else:
            pk = packed.numpy()
            codes = np.empty(pk.shape[:-1] + (pk.shape[-1] * 2,), np.uint8)
            codes[..., 0::2], codes[..., 1::2] = pk & 0xF, pk >> 4
            v = codes.view(ml.float4_e2m1fn).astype(np.float64)
        s = sf.numpy().view(ml.float8_e8m0fnu).astype(np.float64)
        return torch.from_numpy(v * np.repeat(s, 32, axis=-1))

    quant = {MI.QUANT_W4A8: quant, MI.QUANT_W8A8: quant_mx, MI.QUANT_W4A16: no_quant}[mode]
    xd, xs = quant(x)
    I = case.cfg.inter
    out = torch.zeros(T, case.cfg.hidden, dtype=torch.float64)
    for e in range(E):
        G = (xd @ dense(case.w1[e], case.w1_sf[e]).T).to(torch.float32) * xs[:, None].to(torch.float32)
        g, u = G[:, :I], G[:, I:]
        h = (g / (1 + torch.exp(-g)) * u).to(torch.bfloat16).to(torch.float32)
        hd, hs = quant(h)
        Y = (hd @ dense(case.w2[e], case.w2_sf[e]).T).to(torch.float32) * hs[:, None].to(torch.float32)
        out += wsel[:, e:e + 1] * Y.to(torch.float64)
    return out.to(torch.float32).to(torch.bfloat16).to(torch.float32).numpy(), sel


@pytest.mark.parametrize("mode", [MI.QUANT_W4A8, MI.QUANT_W8A8, MI.QUANT_W4A16])
@pytest.mark.parametrize("E,k,H,I,T", [(8, 2, 256, 128, 16), (6, 3, 128, 64, 40),
                                       (4, 4, 64, 32, 9), (16, 1, 128, 96, 23)])
def test_forward_vs_brute_force(E, k, H, I, T, mode):
    cfg = MI.custom_config(E, k, H, I, mode=mode)
    case = MI.make_case(cfg, T, seed=100 + T)
    ref, sel = brute_force(case, k, mode)
    xbits, logits, W = _to_np(case)
    fw = M.forward(xbits, logits, W, k, mode=mode)
    np.testing.assert_array_equal(np.sort(fw.routing.ids, 1),
                                  np.sort(np.nonzero(sel.numpy())[1].reshape(T, k), 1))
    # equal up to the order of the final float64 sum (one bf16 ulp at most)
    diff = np.abs(fw.out - ref)
    assert np.all(diff <= 2.0 ** -8 * np.abs(ref) + 1e-30), diff.max()
    assert diff.sum() <= 1e-6 * np.abs(ref).sum()


def test_forward_token_subset_is_exact():
    cfg = MI.CONFIGS["tiny"]
    case = MI.make_case(cfg, 16)
    xbits, logits, W = _to_np(case)
    full = M.forward(xbits, logits, W, cfg.top_k)
    toks = np.array([3, 0, 11, 15])
    sub = M.forward(xbits, logits, W, cfg.top_k, tokens=toks)
    np.testing.assert_array_equal(sub.out, full.out[toks])


def test_silu_formula_matches_torch():
    z = torch.linspace(-30, 30, 100001, dtype=torch.float32)
    ref = torch.nn.functional.silu(z.double()).float().numpy()
    got = M.silu_f32(z.numpy())
    ulp = np.spacing(np.abs(ref).astype(np.float32))
    assert np.all(np.abs(got - ref) <= 4 * ulp)
