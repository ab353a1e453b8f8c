"""GPU parity of the W4A16 mode (MXFP4 weights x bf16 activations) against
the CPU oracle on the same seeded inputs.  The device carries each bf16
activation (and each element of h) into the FP8 tensor cores as two MXFP8
terms; the oracle's forward is the exact bf16 product.

Bit-exact: routing, expansion, and the two-term codes and scale bytes of
the expanded rows and of h (against the oracle's split of the same bf16
values).  Floating point (h, y, output): max|err| <= 2e-2 * max|ref| and
sum|err| / sum|ref| <= 5e-3."""
import numpy as np
import pytest
import torch

import moe_inputs as MI
import precision_moe_grouped_gb300 as P
from oracle import moe as M

from gpu_helpers import DeviceRun, dump, max_err_ok, oracle_weights, x_bits

pytestmark = pytest.mark.gpu

W4A16 = MI.QUANT_W4A16


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.load()


def w16_parity(case, name="w16"):
    assert case.mode == W4A16
    run = DeviceRun(case)
    assert run.status == 0
    fw = M.forward(x_bits(case), case.logits.cpu().numpy(), oracle_weights(case),
                   case.cfg.top_k, mode=M.QUANT_W4A16)
    rt = fw.routing
    try:
        np.testing.assert_array_equal(run.ids, rt.ids)
        np.testing.assert_array_equal(run.offsets, rt.offsets)
        np.testing.assert_array_equal(run.row_of, rt.row_of)
        np.testing.assert_array_equal(run.token_slot // run.k, rt.token_of_row)
        # the expanded rows: the two-term split of the tokens' bf16 rows
        xc, xs = M.split_rows_mxfp8x2(case.x.float().cpu().numpy()[rt.token_of_row])
        np.testing.assert_array_equal(run.xq, xc)
        np.testing.assert_array_equal(run.x_sf, xs)
        # GEMM2's operand: the split of the GPU's own h
        hc, hs = M.split_rows_mxfp8x2(run.h)
        np.testing.assert_array_equal(run.hq, hc)
        np.testing.assert_array_equal(run.h_sf, hs)
        for label, got, ref in (("h", run.h, fw.h), ("y", run.y, fw.y),
                                ("out", run.out_np(), fw.out)):
            ok, st = max_err_ok(got, ref)
            assert ok, (label, st)
    except AssertionError:
        dump(name, h=run.h, h_ref=fw.h, y=run.y, y_ref=fw.y, out=run.out_np(), out_ref=fw.out,
             tiles=run.tiles)
        raise
    return run, fw


def _cfg(E, k, H, I):
    return MI.custom_config(E, k, H, I, mode=W4A16, name="w16_custom")


def test_w16_tiny():
    w16_parity(MI.make_case(_cfg(8, 2, 256, 128), 16), name="w16_tiny")


def test_w16_ragged_tiles():
    """Several 64-token tiles per expert, ragged tails, several M-tiles and
    K stages."""
    run, _ = w16_parity(MI.make_case(_cfg(8, 2, 512, 256), 300, seed=7), name="w16_ragged")
    assert run.tiles[:, 2].max() <= 64 and run.counts.max() > 64


@pytest.mark.parametrize("E,k,T", [(1, 1, 5), (16, 16, 3), (32, 1, 7)])
def test_w16_degenerate_routing(E, k, T):
    w16_parity(MI.make_case(_cfg(E, k, 128, 128), T, seed=31 + T), name=f"w16_degen{E}_{k}")


def test_w16_zero_rows():
    case = MI.make_case(_cfg(8, 2, 256, 128), 24, seed=41)
    case.x[3] = 0
    case.x[5, 7] = -0.0
    w16_parity(case, name="w16_zeros")


def test_w16_config_full():
    """The W4A16 workload in full: E=64, top-4, H=2048, I=1024, T=256."""
    cfg = MI.CONFIGS["w4a16"]
    w16_parity(MI.make_case(cfg, 256, device="cuda"), name="w16_config")


def test_w16_large_batch_expansion():
    """T > 256: the bf16 rows are copied by the multi-kernel expansion
    (scan, scatter) instead of the one-kernel small-batch path."""
    run, _ = w16_parity(MI.make_case(_cfg(8, 2, 256, 128), 1500, seed=5), name="w16_large")
    assert run.T > P._lib.MOE_SMALL_BATCH_TOKENS


def test_w16_wide_dynamic_range():
    """Rows whose elements span 2^-40 .. 2^8 inside each 32-block, so many
    fall below the split's exact range (2^-13 of the block maximum): the
    codes still match the oracle's split bit for bit, and the outputs stay
    within the tolerance of the exact bf16 product."""
    case = MI.make_case(_cfg(8, 2, 256, 128), 40, seed=17)
    g = torch.Generator().manual_seed(3)
    mag = torch.pow(2.0, torch.randint(-40, 9, case.x.shape, generator=g).float())
    case.x = (case.x.float() * mag).to(torch.bfloat16)
    w16_parity(case, name="w16_wide")
