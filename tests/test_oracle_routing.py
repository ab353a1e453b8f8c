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


def _independent_front(x_bf16: torch.Tensor, logits: torch.Tensor, k: int):
    """Steps 1-3 written with torch primitives only (no oracle routine):
    torch.topk + softmax routing (distinct logits), a stable argsort of the
    flattened expert ids for the expert-major order (ascending token inside
    an expert, since a token's k experts are distinct), and the per-token
    E4M3 codes by torch's float8 cast of x * fl32(448 / amax) clamped to 448."""
    T, E = logits.shape
    _, ids = torch.topk(logits.double(), k, dim=1, sorted=True)
    sel = logits.double().gather(1, ids)
    w = torch.softmax(sel, dim=1)
    flat = ids.reshape(-1)
    order = torch.sort(flat, stable=True).indices          # row r <- flat (t, j)
    row_of = torch.empty_like(order)
    row_of[order] = torch.arange(T * k)
    counts = torch.bincount(flat, minlength=E)
    x = x_bf16.float()
    amax = x.abs().amax(dim=1)
    nz = amax > 0
    safe = torch.where(nz, amax, torch.ones_like(amax))
    inv = torch.tensor(448.0, dtype=torch.float32) / safe
    s = torch.where(nz, safe / torch.tensor(448.0, dtype=torch.float32), torch.ones_like(amax))
    prod = (x * inv[:, None]).clamp(-448.0, 448.0)
    codes = prod.to(torch.float8_e4m3fn).view(torch.uint8)
    codes[~nz] = 0
    return (ids.int().numpy(), w.float().numpy(), counts.int().numpy(),
            row_of.reshape(T, k).int().numpy(), (order // k).int().numpy(), codes.numpy(),
            s.numpy())


def check_route_and_quantize(fn, x_bf16: torch.Tensor, logits: torch.Tensor, k: int):
    """route_and_quantize (the reference the full-size GPU tests take their
    bit-exact front end from) against the independent torch formulation and
    against forward()'s own routing and expanded codes."""
    bits = x_bf16.view(torch.int16).numpy().view(np.uint16)
    lg = logits.numpy()
    rt, tq, ts = fn(bits, lg, k)
    ids, w, counts, row_of, tok_of_row, codes, s = _independent_front(x_bf16, logits, k)
    np.testing.assert_array_equal(rt.ids, ids)
    np.testing.assert_allclose(rt.weights, w, rtol=3e-7, atol=0)
    np.testing.assert_array_equal(rt.counts, counts)
    np.testing.assert_array_equal(rt.row_of, row_of)
    np.testing.assert_array_equal(rt.token_of_row, tok_of_row)
    np.testing.assert_array_equal(tq, codes)
    np.testing.assert_array_equal(ts, s)
    # the same rows forward() quantises and feeds to GEMM1 (W4A8 mode)
    E, H = logits.shape[1], x_bf16.shape[1]
    W = M.Weights(np.zeros((E, 256, H // 2), np.uint8), np.full((E, 256, H // 32), 127, np.uint8),
                  np.zeros((E, H, 64), np.uint8), np.full((E, H, 4), 127, np.uint8))
    fw = M.forward(bits, lg, W, k)
    np.testing.assert_array_equal(tq[rt.token_of_row], fw.xq)
    np.testing.assert_array_equal(ts[rt.token_of_row], fw.x_scale)
    np.testing.assert_array_equal(rt.row_of, fw.routing.row_of)


def _front_cases():
    g = torch.Generator().manual_seed(23)
    # the tiny workload shape: E=8, top-2, H=256, T=16
    x1 = torch.randn(16, 256, generator=g).to(torch.bfloat16)
    l1 = torch.randn(16, 8, generator=g)
    # skewed routing (Zipf(1.2) bias over 64 experts, many empty), rows of
    # widely different magnitude and an all-zero row
    x2 = (torch.randn(40, 512, generator=g) *
          torch.exp(torch.empty(40, 1).uniform_(-8, 8, generator=g))).to(torch.bfloat16)
    x2[7] = 0
    ranks = torch.randperm(64, generator=g).float() + 1
    l2 = torch.randn(40, 64, generator=g) - 1.2 * torch.log(ranks)[None, :]
    return [(x1, l1, 2), (x2, l2, 6)]


@pytest.mark.parametrize("case", [0, 1])
def test_route_and_quantize_matches_independent_front(case):
    x, lg, k = _front_cases()[case]
    check_route_and_quantize(M.route_and_quantize, x, lg, k)
