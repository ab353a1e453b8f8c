"""GPU parity of the MXFP8 x MXFP8 mode (W8A8: E4M3 weights and activations,
one E8M0 scale per 32-element K block on both operands) against the CPU
oracle on the same seeded inputs.

Bit-exact: routing, expansion, the activation E4M3 codes and their E8M0
block-scale bytes (row-major and in the GEMM's per-tile layout).  Floating
point (h, y, output): max|err| <= 2e-2 * max|ref| and
sum|err| / sum|ref| <= 5e-3."""
import numpy as np
import pytest
import torch

import moe_inputs as MI
import precision_moe_grouped_gb300 as P
from oracle import moe as M

from gpu_helpers import DeviceRun, dump, max_err_ok, oracle_weights, x_bits

pytestmark = pytest.mark.gpu

W8A8 = MI.QUANT_W8A8
SFB_TILE_BYTES = 1024


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.load()


def _sfb_offset(n: int) -> int:
    """Byte of tile row n inside a 1024-byte (tile, K stage) block: 32 lanes x
    16 bytes per 128 rows, row 32i + l at 16l + 4i."""
    return (n >> 7) * 512 + 16 * (n & 31) + 4 * ((n >> 5) & 3)


def check_tiled_scales(run: DeviceRun, which: str):
    """The per-tile scale copy holds, for every row of every tile, the same
    bytes as the row-major scales (x: K = H, h: K = I)."""
    K = run.H if which == "x" else run.I
    KS = K // 128
    rowmajor = run.x_sf if which == "x" else run.h_sf
    name = "x_sf_tiled" if which == "x" else "h_sf_tiled"
    tiles = run.tiles
    blob = run.bytes_(name, len(tiles) * KS * SFB_TILE_BYTES)
    for t, (_, r0, nrows, _) in enumerate(tiles):
        for n in range(nrows):
            for ks in range(KS):
                base = (t * KS + ks) * SFB_TILE_BYTES + _sfb_offset(n)
                np.testing.assert_array_equal(blob[base:base + 4],
                                              rowmajor[r0 + n, 4 * ks:4 * ks + 4])


def check_front_mx(run: DeviceRun, rt: M.Routing, tq: np.ndarray, ts: np.ndarray, rows=None):
    np.testing.assert_array_equal(run.ids, rt.ids)
    np.testing.assert_array_equal(run.counts, rt.counts)
    np.testing.assert_array_equal(run.offsets, rt.offsets)
    np.testing.assert_array_equal(run.row_of, rt.row_of)
    ts_gpu = run.token_slot
    np.testing.assert_array_equal(ts_gpu // run.k, rt.token_of_row)
    np.testing.assert_array_equal(ts_gpu % run.k, rt.slot_of_row)
    np.testing.assert_allclose(run.weights, rt.weights, rtol=3e-6, atol=1e-7)
    np.testing.assert_array_equal(run.x_sf, ts[rt.token_of_row])
    sel = np.arange(run.R) if rows is None else np.asarray(rows)
    np.testing.assert_array_equal(run.xq[sel], tq[rt.token_of_row[sel]])


def mx_parity(case, variant=0, name="mx"):
    assert case.mode == W8A8
    run = DeviceRun(case, variant=variant)
    assert run.status == 0
    fw = M.forward(x_bits(case), case.logits.cpu().numpy(), oracle_weights(case),
                   case.cfg.top_k, mode=M.QUANT_W8A8)
    try:
        check_front_mx(run, fw.routing, *M.quantize_rows_mxfp8(
            np.asarray(case.x.float().cpu().numpy(), np.float32)))
        # GEMM2's MXFP8 operand: the oracle's block quantiser applied to the
        # GPU's own h gives the same codes and scale bytes bit for bit
        hq_ref, hsf_ref = M.quantize_rows_mxfp8(run.h.astype(np.float32))
        np.testing.assert_array_equal(run.hq, hq_ref)
        np.testing.assert_array_equal(run.h_sf, hsf_ref)
        for label, got, ref in (("h", run.h, fw.h), ("y", run.y, fw.y),
                                ("out", run.out_np(), fw.out)):
            ok, st = max_err_ok(got, ref)
            assert ok, (label, st)
    except AssertionError:
        dump(name, h=run.h, h_ref=fw.h, y=run.y, y_ref=fw.y, out=run.out_np(), out_ref=fw.out,
             xq=run.xq, xq_ref=fw.xq, x_sf=run.x_sf, x_sf_ref=fw.x_scale, tiles=run.tiles)
        raise
    return run, fw


def _cfg(E, k, H, I, zipf=0.0):
    return MI.custom_config(E, k, H, I, mode=W8A8, zipf=zipf, name="mx_custom")


def test_mx_tiny_full():
    run, _ = mx_parity(MI.make_case(_cfg(8, 2, 256, 128), 16), name="mx_tiny")
    check_tiled_scales(run, "x")
    check_tiled_scales(run, "h")


@pytest.mark.parametrize("variant", [1, 2, 3, 4, 5])
def test_mx_several_tiles_ragged(variant):
    """Several token tiles per expert, ragged tails, several weight M-tiles
    and K stages, every tile variant."""
    run, _ = mx_parity(MI.make_case(_cfg(8, 2, 512, 256), 200, seed=7), variant=variant,
                       name=f"mx_ragged{variant}")
    check_tiled_scales(run, "x")


@pytest.mark.parametrize("variant", [2, 4, 5])
def test_mx_tiles_over_128_rows(variant):
    """Tiles of more than 128 rows: the activation scales of MMA-N rows
    128.. come from the second 512-byte half of each per-tile block."""
    # ~150 rows per expert: one tile of 129..160 rows in every variant listed
    run, _ = mx_parity(MI.make_case(_cfg(4, 2, 256, 128), 300, seed=9), variant=variant,
                       name=f"mx_split{variant}")
    assert run.tiles[:, 2].max() > 128
    check_tiled_scales(run, "h")


def test_mx_zipf_skew_with_empty_experts():
    """Zipf(1.2)-biased routing (the MXFP8 workload's skew): hot experts get
    many rows, some experts none."""
    run, fw = mx_parity(MI.make_case(_cfg(64, 8, 256, 256, zipf=1.2), 96, seed=17),
                        name="mx_zipf")
    counts = run.counts
    assert (counts == 0).any() and counts.max() >= 4 * counts.mean()


def test_mx_variants_agree_bitwise():
    case = MI.make_case(_cfg(8, 2, 256, 128), 96, seed=13)
    a = DeviceRun(case, variant=1)
    for v in (2, 3, 4, 5):
        b = DeviceRun(case, variant=v, moe=a.moe)
        np.testing.assert_array_equal(a.out_np(), b.out_np())


def test_mx_zero_and_tiny_blocks():
    """An all-zero token, an all-zero block holding -0.0 (scale byte 127,
    codes of +-0) and a block of subnormal-range values next to a large one."""
    case = MI.make_case(_cfg(8, 2, 256, 128), 24, seed=41)
    case.x[3] = 0
    case.x[5, 32:64] = 0
    case.x[5, 40] = -0.0
    case.x[7, 0:32] = 1e-30
    case.x[7, 3] = 3.0e4
    run, fw = mx_parity(case, name="mx_zeros")
    r = run.row_of[3, 0]
    assert (run.x_sf[r] == 127).all() and (run.xq[r] == 0).all()


@pytest.mark.parametrize("T", [4096])
def test_mx_zipf_full_size(T):
    """The MXFP8 workload at full size (E=256, top-8, H=7168, I=2048,
    Zipf 1.2, T=4096) in the bench's launch configuration: routing,
    expansion, the codes and the block-scale bytes bit-exact on every row,
    the output on a token sample."""
    cfg = MI.CONFIGS["mxfp8_zipf"]
    case = MI.make_case(cfg, T, device="cuda")
    run = DeviceRun(case)
    assert run.status == 0
    x32 = np.asarray(case.x.float().cpu().numpy(), np.float32)
    ids, w = M.route(case.logits.cpu().numpy(), cfg.top_k)
    rt = M.expand(ids, w, cfg.num_experts)
    tq, ts = M.quantize_rows_mxfp8(x32)
    check_front_mx(run, rt, tq, ts)     # every expanded row's codes and scale bytes
    rng = np.random.default_rng(T)
    assert (run.counts == 0).any()
    toks = np.sort(rng.choice(T, size=3, replace=False))
    fw = M.forward(x_bits(case), case.logits.cpu().numpy(), oracle_weights(case), cfg.top_k,
                   mode=M.QUANT_W8A8, tokens=toks)
    ok, st = max_err_ok(run.out_np()[toks], fw.out)
    if not ok:
        dump(f"mxfp8_zipf_{T}", out=run.out_np()[toks], out_ref=fw.out, toks=toks)
    assert ok, st
