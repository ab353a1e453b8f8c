"""GPU parity of the CTA-pair grouped GEMM (tile variant 6: two SMs share
each 256-row tcgen05 MMA, each staging half of the token tile) against the
CPU oracle, with the same bars as the one-CTA kernel: bit-exact routing,
expansion and FP8 codes; h, y and the output within max|err| <=
2e-2 * max|ref| and sum|err| / sum|ref| <= 5e-3."""
import numpy as np
import pytest
import torch

import moe_inputs as MI
import precision_moe_grouped_gb300 as P

from gpu_helpers import DeviceRun
from test_gpu_parity import _sampled_parity, check_tiles, full_parity

pytestmark = pytest.mark.gpu

PAIR = 6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.load()


def test_pair_small_full():
    """One pair item per tile (2I = H = 256: two M-tiles), ragged tiles."""
    cfg = MI.custom_config(8, 2, 256, 128)
    run, _ = full_parity(MI.make_case(cfg, 90, seed=3), variant=PAIR, name="pair_small")
    check_tiles(run, 160)


def test_pair_several_items_and_stages():
    """Several M-tile pairs per tile (2I = H = 512), several K stages, more
    pipeline fills per CTA than slots."""
    cfg = MI.custom_config(8, 2, 512, 256)
    full_parity(MI.make_case(cfg, 200, seed=7), variant=PAIR, name="pair_ragged")


def test_pair_tiles_split_and_tails():
    """Experts with more rows than a tile: balanced tiles of <= 160 rows,
    token counts that are not multiples of 32 (the MMA's N rounds up)."""
    cfg = MI.custom_config(4, 2, 256, 128)
    run, _ = full_parity(MI.make_case(cfg, 700, seed=9), variant=PAIR, name="pair_split")
    assert run.counts.max() > 160
    assert (run.tiles[:, 2] % 32 != 0).any()
    check_tiles(run, 160)


def test_pair_odd_m_tiles_fall_back():
    """H = 384: GEMM2 has three M-tiles, so it runs on the one-CTA kernel
    while GEMM1 (2I = 256) runs on pairs; both must match the oracle."""
    cfg = MI.custom_config(8, 2, 384, 128)
    full_parity(MI.make_case(cfg, 64, seed=11), variant=PAIR, name="pair_odd")


def test_pair_small_tiles():
    """Tiles of 1..31 rows: the smallest pair MMA (N = 32, 16 rows per CTA)."""
    cfg = MI.custom_config(32, 2, 256, 256)
    run, _ = full_parity(MI.make_case(cfg, 40, seed=13), variant=PAIR, name="pair_tiny_tiles")
    assert run.tiles[:, 2].max() <= 31


def test_pair_matches_one_cta_kernel():
    """The pair kernel and the one-CTA kernel with the same tiles (variant
    5) compute the same products; their outputs agree to bf16 rounding."""
    cfg = MI.custom_config(8, 2, 512, 256)
    case = MI.make_case(cfg, 150, seed=17)
    a = DeviceRun(case, variant=5)
    b = DeviceRun(case, variant=PAIR, moe=a.moe)
    np.testing.assert_array_equal(a.tiles, b.tiles)
    diff = np.abs(a.out_np().astype(np.float64) - b.out_np().astype(np.float64))
    assert diff.max() <= 1e-2 * np.abs(a.out_np().astype(np.float64)).max()


def test_pair_deterministic():
    cfg = MI.custom_config(16, 4, 256, 256)
    case = MI.make_case(cfg, 300, seed=21)
    a = DeviceRun(case, variant=PAIR)
    b = DeviceRun(case, variant=PAIR, moe=a.moe)
    np.testing.assert_array_equal(a.out_np(), b.out_np())


@pytest.mark.parametrize("T", [512, 4096])
def test_pair_dsv3_sizes(T):
    """The DSV3 layer (E=256, top-8, H=7168, I=2048) at prefill sizes on
    pairs: front end bit-exact on every token, output on a token sample."""
    _sampled_parity(MI.CONFIGS["dsv3"], T, n_sample=4, variant=PAIR)
