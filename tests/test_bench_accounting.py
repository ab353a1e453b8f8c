"""bench.py's roofline accounting, checked against sizes written out by hand
for the DSV3 layer (E=256, top-8, H=7168, I=2048) in each quantisation
mode: the algorithmic bytes and flops of one GEMM launch and of the whole
forward, and which tensor peak each mode is held to."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_inputs as MI  # noqa: E402

E, K, H, I, T = 256, 8, 7168, 2048, 4096
R = T * K
PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}


def test_gemm_bytes_per_mode():
    cfg = MI.CONFIGS["dsv3"]
    # W4A8: packed E2M1 (half a byte) + one E8M0 byte per 32; FP8 rows + row scale
    b, f = bench.alg_cost("gemm1", cfg, T, E, mode=0)
    assert b == E * 2 * I * H * (0.5 + 1 / 32) + R * H + R * 4 + R * I * 2
    assert f == 2.0 * R * H * 2 * I
    # W8A8: E4M3 weights, activations with one scale byte per 32, no row scale
    b, f = bench.alg_cost("gemm2", cfg, T, E, mode=2)
    assert b == E * H * I * (1 + 1 / 32) + R * I * (1 + 1 / 32) + R * H * 2
    assert f == 2.0 * R * I * H
    # W4A16: each bf16 activation (and element of h) as two E4M3 terms, each
    # term with one scale byte per 32; no row scale
    b, _ = bench.alg_cost("gemm1", cfg, T, E, mode=1)
    assert b == E * 2 * I * H * (0.5 + 1 / 32) + R * H * (2 + 2 / 32) + R * I * 2
    b, _ = bench.alg_cost("hquant", cfg, T, E, mode=1)
    assert b == R * I * 2 + R * I * (2 + 2 / 32)


@pytest.mark.parametrize("mode,w_bytes,peak", [(0, 0.5, 2 * 2000.0), (1, 0.5, 2000.0),
                                               (2, 1.0, 2 * 2000.0)])
def test_fused_roofline_per_mode(mode, w_bytes, peak):
    cfg = MI.CONFIGS["dsv3"]
    fr = bench.fused_roofline(cfg, T, E, 1e-3, PEAKS, mode)
    weights = E * 3 * I * H * (w_bytes + 1 / 32)
    io = T * H * 2 + T * E * 4 + T * H * 2          # x in, logits in, out
    assert fr["bytes"] == pytest.approx(weights + io)
    assert fr["flops"] == 2.0 * T * K * 3 * I * H
    assert fr["t_hbm_us"] == pytest.approx((weights + io) / 8000e9 * 1e6)
    assert fr["t_tensor_us"] == pytest.approx(2.0 * T * K * 3 * I * H / (peak * 1e12) * 1e6)
    # the larger of the two times sets the bound: HBM for the FP8 MMA kinds,
    # the tensor pipe for bf16 (W4A16 would be compute-bound at this size)
    assert fr["bound"] == ("tensor" if mode == 1 else "hbm")
    assert fr["frac"] == pytest.approx(max(fr["t_hbm_us"], fr["t_tensor_us"]) / 1e3)


def test_touched_experts_scale_the_weight_bytes():
    cfg = MI.CONFIGS["dsv3"]
    one = bench.fused_roofline(cfg, 1, 8, 1e-3, PEAKS)["bytes"]
    assert one == pytest.approx(8 * 3 * I * H * (0.5 + 1 / 32) + H * 2 + E * 4 + H * 2)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_oracle_cost_parts_reproduce_forward(mode):
    """The timed parts of the CPU baseline run the oracle's own steps: the
    token-linear part and every expert's part together reproduce forward()'s
    routing and y rows bit for bit, so timing them times the forward."""
    import numpy as np
    import torch

    from oracle import moe as M
    cfg = MI.custom_config(8, 2, 256, 128, mode=mode)
    case = MI.make_case(cfg, 24, seed=5)
    xb = case.x.view(torch.int16).numpy().view(np.uint16)
    lg = case.logits.numpy()
    W = M.Weights(case.w1.numpy(), case.w1_sf.numpy(), case.w2.numpy(), case.w2_sf.numpy(),
                  mode=mode)
    fw = M.forward(xb, lg, W, cfg.top_k, mode=mode)
    rt, a1, xs, _ = bench.oracle_token_part(xb, lg, cfg.top_k, cfg.num_experts, mode)
    np.testing.assert_array_equal(rt.row_of, fw.routing.row_of)
    for e in range(cfg.num_experts):
        r0, r1 = int(rt.offsets[e]), int(rt.offsets[e + 1])
        if r1 == r0:
            continue
        y = bench.oracle_expert_part(W, e, a1[r0:r1], None if xs is None else xs[r0:r1], mode)
        np.testing.assert_array_equal(y, fw.y[r0:r1])


def test_cpu_baseline_extrapolates_from_timed_parts():
    """t(T) = T * t_token + n_touched * t_expert, reported as extrapolated."""
    cfg = MI.CONFIGS["tiny"]
    case = MI.make_case(cfg, 16)
    res = bench.cpu_baseline(cfg, 16, case.x, case.logits, n_tok=8, n_exp=2)
    assert res["extrapolated"] and res["kind"] == "oracle"
    assert res["value"] == pytest.approx(16 / res["t_forward_s"])
    assert "extrapolated" in res["sample"]
