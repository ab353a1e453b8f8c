"""Exact CPU codecs for the number formats of the fused MXFP4 MoE forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.

Pages cited (title and section):
  [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
          MXFP4xFP8 CUTLASS MoE backend for SM90", Description and
          Implementation Notes (MXFP4 weight = E2M1 values with one E8M0 scale;
          FP8 activations).
  [P4793] flashinfer PR #4793, "Unify MoE CuTe DSL dispatch to be dtype
          agnostic", review comments (scale tensors are uint8 E8M0 bytes).
  [P3614] flashinfer PR #3614, "fix: make the cutlass MoE gemm profiler
          MXFP8-aware", discussion (biased exponent 0x7F encodes 1.0).

The pages name the formats but do not define their bit layouts.  The bit
layouts below are the OCP Microscaling (MX) v1.0 definitions:
  E2M1  sign | 2-bit exponent (bias 1) | 1-bit mantissa, no Inf/NaN, max 6.
  E4M3  sign | 4-bit exponent (bias 7) | 3-bit mantissa, no Inf, NaN at
        S.1111.111, max 448, subnormals 2^-6 * m/8.
  E8M0  8-bit unsigned biased exponent, value 2^(b-127), 0xFF is NaN.
  bf16  upper half of an IEEE binary32.

Every function is written from those definitions with float64 arithmetic
(which holds every value of these formats exactly).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _e2m1_value(c: np.ndarray) -> np.ndarray:
    """OCP MX E2M1 definition applied to 4-bit codes."""
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    exp = ((c >> 1) & 3).astype(np.int64)
    man = (c & 1).astype(np.float64)
    # exponent field 0 is subnormal: 2^(1-bias) * (m/2) with bias 1
    mag = np.where(exp == 0, man * 0.5, np.ldexp(1.0 + man * 0.5, exp - 1))
    return sign * mag


def _e4m3_value(c: np.ndarray) -> np.ndarray:
    """OCP MX E4M3 (fn variant) definition applied to 8-bit codes."""
    c = c.astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = (c & 7).astype(np.float64)
    mag = np.where(exp == 0,
                   np.ldexp(man / 8.0, -6),
                   np.ldexp(1.0 + man / 8.0, exp - 7))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def _e8m0_value(b: np.ndarray) -> np.ndarray:
    """OCP MX E8M0 definition: 2^(b-127), 0xFF is NaN."""
    b = b.astype(np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


# The definitions above are evaluated once for every code; decoding a tensor
# is then a table lookup (same values, without per-element exponent work).
_E2M1_TABLE = _e2m1_value(np.arange(16, dtype=np.uint8))
_E4M3_TABLE = _e4m3_value(np.arange(256, dtype=np.uint8))
_E8M0_TABLE = _e8m0_value(np.arange(256, dtype=np.uint8))


def e2m1_decode(codes) -> np.ndarray:
    """Value of each 4-bit E2M1 code (low nibble of each uint8), float64."""
    return _E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def e8m0_decode(codes) -> np.ndarray:
    """Value 2^(b-127) of each E8M0 byte, float64; 0xFF decodes to NaN."""
    return _E8M0_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 (fn variant) byte, float64; 0x7F/0xFF are NaN."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(values) -> np.ndarray:
    """E4M3 code of each value, round-to-nearest-even, saturating to +-448.

    ``values`` are taken as given (float32 inputs are widened exactly).  The
    sign bit of the input is kept, so -0.0 and negative values that round to
    zero give 0x80.  NaN gives 0x7F with its sign.  This is the conversion an
    IEEE-style 'round to nearest even, satfinite' cast performs.
    """
    v = np.asarray(values, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # below the smallest normal 2^-6 the grid is uniform with step 2^-9
    sub = a < 2.0 ** -6
    q_sub = np.rint(a * 2.0 ** 9)          # rint = round half to even
    code_sub = q_sub.astype(np.int64)       # 8 carries into exponent 1
    # normal range: a = 2^e * (q/8) with q in [8, 16)
    safe = np.where(sub | (a == 0), 1.0, a)
    _, e2 = np.frexp(safe)                  # safe = f * 2^e2, f in [0.5, 1)
    e = e2 - 1
    q = np.rint(np.ldexp(safe, 3 - e))      # exact scaling, then RNE
    code_norm = ((e + 7) << 3) + (q.astype(np.int64) - 8)  # q == 16 carries
    code = np.where(sub, code_sub, code_norm)
    code = np.minimum(code, 0x7E)           # satfinite: overflow -> 448
    code = np.where(nan, 0x7F, code)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def bf16_round(values) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns
    the rounded values as float32.  Finite inputs only."""
    f = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """float32 value of raw bf16 bit patterns (uint16)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f32_to_bf16_bits(values) -> np.ndarray:
    """bf16 bit pattern (uint16) of float32 values, rounding to nearest even."""
    r = bf16_round(values)
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """Split packed E2M1 bytes [..., K/2] into codes [..., K].

    Byte j of a row holds element 2j in its low nibble and element 2j+1 in its
    high nibble (little-endian nibble order; the pages fix K = 2 x the byte
    width of the weight tensor but not the nibble order)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def mxfp4_dequant(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dense float64 matrix of an MXFP4 tensor.

    ``packed`` uint8 [..., N, K/2] (two E2M1 codes per byte), ``scales`` uint8
    [..., N, K/32] (one E8M0 byte per 32 consecutive K elements of a row)
    [P3738 Description; P4793 review comments].  Element (n, k) is
    E2M1(n, k) * 2^(scale(n, k // 32) - 127)."""
    p = np.asarray(packed, dtype=np.uint8)
    # value pair of every possible byte, through the same unpack + decode
    pair = e2m1_decode(unpack_e2m1(np.arange(256, dtype=np.uint8)[:, None]))   # [256, 2]
    vals = pair[p].reshape(p.shape[:-1] + (p.shape[-1] * 2,))
    sc = e8m0_decode(scales)
    blk = vals.reshape(vals.shape[:-1] + (vals.shape[-1] // 32, 32))
    return (blk * sc[..., None]).reshape(vals.shape)


def mxfp8_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dense float64 matrix of an MXFP8 (E4M3 + E8M0 per 32) tensor."""
    vals = e4m3_decode(codes)
    sc = e8m0_decode(scales)
    return vals * np.repeat(sc, 32, axis=-1)
