"""Pins of the oracle's routing, expansion and FP8 quantiser against
torch.topk / softmax, counting invariants and the quantiser's error bound."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import moe as M


def test_route_matches_torch_topk_softmax():
    g = torch.Generator().manual_seed(11)
    for (T, E, k) in [(64, 8, 2), (33, 256, 8), (17, 384, 6), (5, 16, 16)]:
        logits = torch.randn(T, E, generator=g)
        ids, w = M.route(logits.numpy(), k)
        vals, ref_ids = torch.topk(logits.double(), k, dim=1, sorted=True)
        np.testing.assert_array_equal(ids, ref_ids.numpy())
        ref_w = torch.softmax(logits.double(), dim=1).gather(1, ref_ids)
        ref_w = ref_w / ref_w.sum(dim=1, keepdim=True)
        np.testing.assert_allclose(w, ref_w.numpy(), rtol=2e-7, atol=0)


def test_route_ties_lower_index_first():
    logits = np.array([[1.0, 3.0, 3.0, 0.0, 3.0],
                       [0.0, 0.0, 0.0, 0.0, 0.0],
                       [-0.0, 0.0, -1.0, 2.0, 2.0]], dtype=np.float32)
    ids, w = M.route(logits, 3)
    np.testing.assert_array_equal(ids, [[1, 2, 4], [0, 1, 2], [3, 4, 0]])
    np.testing.assert_allclose(w[0], [1 / 3] * 3, rtol=1e-7)
    np.testing.assert_allclose(w[1], [1 / 3] * 3, rtol=1e-7)


def test_route_weights_sum_to_one_and_ids_distinct():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((500, 64)).astype(np.float32) * 4
    ids, w = M.route(logits, 4)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 4 * 2.0 ** -24 * 4)
    assert all(len(set(r)) == 4 for r in ids.tolist())
    assert np.all(np.diff(w, axis=1) <= 0)             # descending weights


def test_expand_invariants_and_roundtrip():
    rng = np.random.default_rng(4)
    T, E, k = 300, 32, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 5] -= 100.0                                # expert 5 never chosen
    ids, w = M.route(logits, k)
    rt = M.expand(ids, w, E)
    np.testing.assert_array_equal(rt.counts, np.bincount(ids.ravel(), minlength=E))
    assert rt.counts[5] == 0
    assert rt.offsets[0] == 0 and rt.offsets[-1] == T * k
    assert np.all(np.diff(rt.offsets) == rt.counts)
    # permute then un-permute is the identity on (token, slot)
    r = rt.row_of.ravel()
    assert sorted(r.tolist()) == list(range(T * k))
    np.testing.assert_array_equal(rt.token_of_row[rt.row_of], np.repeat(np.arange(T)[:, None], k, 1))
    np.testing.assert_array_equal(rt.slot_of_row[rt.row_of], np.tile(np.arange(k), (T, 1)))
    np.testing.assert_array_equal(rt.expert_of_row[rt.row_of], ids)
    # stable: inside each expert, tokens ascend
    for e in range(E):
        seg = rt.token_of_row[rt.offsets[e]:rt.offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_fp8_quant_bounds_and_amax_code():
    rng = np.random.default_rng(5)
    rows = (rng.standard_normal((64, 512)) * np.exp(rng.uniform(-6, 6, (64, 1)))).astype(np.float32)
    rows[3] = 0.0
    codes, s = M.quantize_rows_fp8(rows)
    assert s[3] == 1.0 and np.all(codes[3] == 0)
    deq = F.e4m3_decode(codes) * s[:, None].astype(np.float64)
    x = rows.astype(np.float64)
    amax = np.abs(x).max(1)
    for i in range(64):
        if i == 3:
            continue
        j = np.argmax(np.abs(x[i]))
        assert codes[i, j] & 0x7F == 0x7E                  # amax element -> +-448
        normal = np.abs(x[i]) >= amax[i] * 2.0 ** -6 / 448 * 1.0001
        err = np.abs(deq[i] - x[i])
        assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[i][normal]) * (1 + 1e-6))
        # below the normal range the absolute step is 2^-9 * s; error <= half
        assert np.all(err[~normal] <= 2.0 ** -10 * s[i] * (1 + 1e-6))


def test_fp8_quant_scale_is_ieee_fp32_division():
    rows = np.array([[3.0, -1.0], [1e-3, 2e-3], [448.0, 1.0]], dtype=np.float32)
    _, s = M.quantize_rows_fp8(rows)
    want = (torch.tensor([3.0, 2e-3, 448.0], dtype=torch.float32) / 448.0).numpy()
    np.testing.assert_array_equal(s, want)


def test_mxfp8_quant_bounds():
    rng = np.random.default_rng(6)
    rows = (rng.standard_normal((8, 256)) * 3).astype(np.float32)
    codes, sc = M.quantize_rows_mxfp8(rows)
    deq = F.mxfp8_dequant(codes, sc)
    x = rows.astype(np.float64)
    X = np.repeat(np.ldexp(1.0, sc.astype(np.int64) - 127), 32, axis=1)
    err = np.abs(deq - x)
    # the block scale puts amax/X in [256, 512): values above 448 X saturate
    # to 448 X (OCP MX v1.0 conversion); the rest carry E4M3's 2^-4 relative
    # rounding bound, or half the 2^-9 X subnormal step
    sat = np.abs(x) > 448 * X
    assert np.all(err[sat] == np.abs(x[sat]) - 448 * X[sat])
    ok = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * X) * (1 + 1e-9)
    assert np.all(err[~sat] <= ok[~sat])
    assert np.all(sc[np.abs(x).reshape(8, 8, 32).max(-1) > 0] > 0)
