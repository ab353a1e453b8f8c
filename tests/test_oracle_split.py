"""Pins of the two-term MXFP8 split (oracle.moe.split_rows_mxfp8x2), the
W4A16 mode's device encoding of bf16 activations: a block worked out by
hand, exact reconstruction over every bf16 value of a 14-binade range,
the error bound below it, no saturation, and zero blocks.  None of these
re-types the function's formula: they check what the two terms must add up
to."""
import numpy as np

from oracle import formats as F
from oracle import moe as M


def _reconstruct(codes, scales):
    """dec(hi) * Xh + dec(lo) * Xl per element, float64, [..., K]."""
    K = codes.shape[-1] // 2
    nb = K // 32
    val = F.e4m3_decode(codes).reshape(codes.shape[:-1] + (2 * nb, 32))
    sc = F.e8m0_decode(scales)[..., None]
    both = (val * sc).reshape(codes.shape[:-1] + (2, K))
    return both[..., 0, :] + both[..., 1, :]


def _bf16(a):
    return F.bf16_round(np.asarray(a, dtype=np.float32))


def test_split_hand_worked_block():
    """Block (1 + 2^-7, 3, -0.5, 0, ...): amax = 3, floor(log2 3) = 1, so
    Xh = 2^(1-7) = 2^-6 (byte 121).  Quotients: 64.5 -> 64 (E4M3 spacing 8
    in [64, 128); code (6+7)<<3 = 0x68), 192 = 1.5 * 2^7 (code (7+7)<<3 + 4
    = 0x74), -32 = -2^5 (code 0x80 | (5+7)<<3 = 0xE0).  Residuals: 2^-7,
    0, 0, so Xl = 2^(-7-7) = 2^-14 (byte 113) and 2^-7 / 2^-14 = 128 = 2^7
    (code 0x70); the other lo codes are +0."""
    x = np.zeros((1, 32), np.float32)
    x[0, :3] = [1.0078125, 3.0, -0.5]
    codes, scales = M.split_rows_mxfp8x2(x)
    assert codes.shape == (1, 64) and scales.shape == (1, 2)
    assert list(codes[0, :3]) == [0x68, 0x74, 0xE0]
    assert not codes[0, 3:32].any()
    assert codes[0, 32] == 0x70 and not codes[0, 33:].any()
    assert list(scales[0]) == [121, 113]


def test_split_exact_over_every_bf16_value_of_14_binades():
    """Every positive and negative bf16 value in [2^-13, 2), in blocks whose
    largest element is 1.9921875 (E = 0): the two terms add up to the value
    exactly."""
    bits = np.arange(0x3900, 0x4000, dtype=np.uint32)        # 2^-13 .. 1.9921875
    vals = F.bf16_bits_to_f32(bits.astype(np.uint16))
    vals = np.concatenate([vals, -vals])
    n = -(-vals.size // 31) * 31
    vals = np.concatenate([vals, np.full(n - vals.size, 0.75, np.float32)])
    rows = np.concatenate([np.full((n // 31, 1), 1.9921875, np.float32),
                           vals.reshape(-1, 31)], axis=1)
    codes, scales = M.split_rows_mxfp8x2(rows)
    np.testing.assert_array_equal(_reconstruct(codes, scales), rows.astype(np.float64))


def test_split_error_bound_and_no_saturation():
    """Random bf16 rows spanning 2^-30 .. 2^12 within a block: elements with
    |v| >= 2^(E-13) reconstruct exactly, the rest within 2^(E-21) (E =
    floor(log2 amax) of the block); every decoded term is at most 256 in
    magnitude (a quotient below 256 may round up to 256, far from the 448
    where E4M3 saturates)."""
    rng = np.random.default_rng(5)
    mag = np.ldexp(1.0, rng.integers(-30, 13, size=(64, 256)))
    x = _bf16(rng.standard_normal((64, 256)) * mag)
    x[3, 40:72] = 0.0
    codes, scales = M.split_rows_mxfp8x2(x)
    rec = _reconstruct(codes, scales)
    blk = x.astype(np.float64).reshape(64, 8, 32)
    amax = np.abs(blk).max(-1, keepdims=True)
    E = np.floor(np.log2(np.where(amax > 0, amax, 1.0))).astype(np.int64)
    err = np.abs(rec.reshape(64, 8, 32) - blk)
    big = np.abs(blk) >= np.ldexp(1.0, E - 13)
    assert (err[big] == 0).all()
    assert (err <= np.ldexp(1.0, E - 21)).all()
    assert (np.abs(F.e4m3_decode(codes)) <= 256).all()


def test_split_zero_block_and_signed_zero():
    """An all-zero block: both scale bytes 0x7F; -0.0 keeps its sign in hi
    (0x80) and leaves a +0 residual (lo code 0x00)."""
    x = np.zeros((1, 64), np.float32)
    x[0, 5] = -0.0
    x[0, 32:] = _bf16(np.linspace(-1, 1, 32))
    codes, scales = M.split_rows_mxfp8x2(x)
    assert scales[0, 0] == 127 and scales[0, 2] == 127
    assert codes[0, 5] == 0x80 and codes[0, 64 + 5] == 0x00
    np.testing.assert_array_equal(_reconstruct(codes, scales)[0], x[0].astype(np.float64))
