"""Plain CPU oracle of the fused MXFP4 x FP8 mixture-of-experts forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA path.

Pages cited (title and section):
  [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
          MXFP4xFP8 CUTLASS MoE backend for SM90": Description (runtime
          activation expansion and per-token FP8 quantization; per-token scale
          epilogue), Implementation Notes (per-token scales computed while
          expanding routed MoE rows; activation token scale applied in the
          epilogue), review comments (fc1/fc2 token scales in the FP8 x MXFP4
          quant params; the activation kernel between the GEMMs).
  [P4793] flashinfer PR #4793, "Unify MoE CuTe DSL dispatch to be dtype
          agnostic": walkthrough (gather grouped GEMM with activation fusion;
          grouped GEMM with finalize fusion; SwiGLU activation).
  [P3614] flashinfer PR #3614, "fix: make the cutlass MoE gemm profiler
          MXFP8-aware": description (MXFP8 x MXFP8 = E4M3 values with E8M0
          block scales on both operands).

The forward, for T tokens, E experts, top-k routing, hidden H, intermediate I:
  1. route:    top-k experts per token from router logits, softmax over the
               k selected logits (renormalised softmax).
  2. expand:   per-expert counts, exclusive-scan offsets, expert-major row
               order with rows of one expert in ascending token order.
  3. quantise: per token, s = amax/448 and E4M3 codes of x * (448/amax).
  4. GEMM1:    g[r, n] = s_t * sum_k dec(xq[r, k]) * dec(w1[e, n, k]),
               w1 rows 0..I-1 = gate, I..2I-1 = up.
  5. SwiGLU:   h = silu(gate) * up, rounded to bf16.
  6. h-quant:  per row, the same FP8 quantiser as step 3.
  7. GEMM2:    y[r, c] = s2_r * sum_j dec(hq[r, j]) * dec(w2[e, c, j]).
  8. combine:  out[t] = sum_j w[t, j] * y[row(t, j)], rounded to bf16.
Dot products are computed in float64; for these formats and sizes every
partial sum is exactly representable, so the float64 result is the exact dot
product, which is then rounded once to float32 (the accumulator precision).
Steps that turn floating point into codes (3, 5, 6) work in float32 as the
kernels do.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import formats as F

QUANT_W4A8 = 0      # MXFP4 weights, per-token FP8 E4M3 activations
QUANT_W4A16 = 1     # MXFP4 weights, bf16 activations
QUANT_W8A8 = 2      # MXFP8 weights and MXFP8 activations


@dataclass
class Routing:
    ids: np.ndarray          # int32 [T, k] expert of slot j, by descending logit
    weights: np.ndarray      # float32 [T, k] renormalised softmax weights
    counts: np.ndarray       # int32 [E]
    offsets: np.ndarray      # int32 [E + 1] exclusive scan of counts
    row_of: np.ndarray       # int32 [T, k] expanded row of (t, j)
    token_of_row: np.ndarray  # int32 [R] token of each expanded row
    slot_of_row: np.ndarray  # int32 [R] slot j of each expanded row
    expert_of_row: np.ndarray  # int32 [R]


def route(logits: np.ndarray, top_k: int) -> tuple[np.ndarray, np.ndarray]:
    """Step 1: top-k softmax routing, renormalised over the selected experts.

    Experts are ranked by raw logit, larger first; equal logits rank the lower
    expert index first (the pages fix no tie rule).  The weights are
    w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the k selected
    logits, i.e. the softmax over all experts renormalised to the top k
    (routing is only implied by the pages' 'routed MoE rows' [P3738
    Implementation Notes]; the rule is the one the workload configuration
    names: top-k softmax routing, renormalised)."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.broadcast_to(np.arange(E), (T, E))
    # lexsort sorts by the last key first: primary -logit, secondary index
    order = np.lexsort((idx, -logits.astype(np.float64)), axis=-1)
    ids = order[:, :top_k].astype(np.int32)
    sel = np.take_along_axis(logits, ids, axis=1).astype(np.float64)
    ex = np.exp(sel - sel.max(axis=1, keepdims=True))
    w = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


def expand(ids: np.ndarray, weights: np.ndarray, num_experts: int) -> Routing:
    """Step 2: expert-major expansion of the routed (token, slot) pairs.

    Rows of expert e occupy [offsets[e], offsets[e+1]); inside one expert the
    rows are in ascending token order [P3738 Description: runtime activation
    expansion of routed MoE rows]."""
    T, k = ids.shape
    counts = np.bincount(ids.ravel(), minlength=num_experts).astype(np.int32)
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    R = int(offsets[-1])
    row_of = np.empty((T, k), dtype=np.int32)
    token_of_row = np.empty(R, dtype=np.int32)
    slot_of_row = np.empty(R, dtype=np.int32)
    expert_of_row = np.empty(R, dtype=np.int32)
    nxt = offsets[:-1].copy()
    for t in range(T):                      # ascending token order
        for j in range(k):
            e = int(ids[t, j])
            r = int(nxt[e])
            nxt[e] += 1
            row_of[t, j] = r
            token_of_row[r] = t
            slot_of_row[r] = j
            expert_of_row[r] = e
    return Routing(ids=ids.astype(np.int32), weights=weights, counts=counts,
                   offsets=offsets.astype(np.int32), row_of=row_of,
                   token_of_row=token_of_row, slot_of_row=slot_of_row,
                   expert_of_row=expert_of_row)


def quantize_rows_fp8(rows_f32: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Steps 3 and 6: per-row FP8 E4M3 quantisation with one float32 scale.

    For a row with amax = max|v| > 0: s = fl32(amax / 448), inv =
    fl32(448 / amax), code = E4M3_rne_satfinite(fl32(v * inv)).  A row whose
    amax is 0 gets s = 1 and all codes 0x00.  Dequantised value = dec(code)*s.
    [P3738 Description and Implementation Notes: runtime per-token FP8
    activation quantization computing per-token scales while expanding rows;
    review comments: fc1/fc2 token scales.]  The pages do not spell out the
    scale rule; amax/448 maps each row's largest magnitude to E4M3's max."""
    v = np.asarray(rows_f32, dtype=np.float32)
    amax = np.max(np.abs(v), axis=-1) if v.shape[-1] else np.zeros(v.shape[:-1], np.float32)
    amax = amax.astype(np.float32)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1.0)).astype(np.float32)
    s = np.where(nz, safe / np.float32(E4M3_MAX_F32), np.float32(1.0)).astype(np.float32)
    inv = (np.float32(E4M3_MAX_F32) / safe).astype(np.float32)
    prod = (v * inv[..., None]).astype(np.float32)
    codes = F.e4m3_encode(prod)
    codes = np.where(nz[..., None], codes, np.uint8(0)).astype(np.uint8)
    return codes, s


E4M3_MAX_F32 = np.float32(F.E4M3_MAX)


def quantize_rows_mxfp8(rows_f32: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """MXFP8 activation quantisation (the W8A8 mode): per 32-element block,
    X = 2^clamp(floor(log2 amax) - 8, -127, 127) (8 = E4M3's emax), codes =
    E4M3_rne_satfinite(v / X); an all-zero block gets scale byte 0x7F
    [P3614 description: MXFP8 x MXFP8 block scales; OCP MX v1.0 conversion]."""
    v = np.asarray(rows_f32, dtype=np.float32).astype(np.float64)
    shp = v.shape
    blk = v.reshape(shp[:-1] + (shp[-1] // 32, 32))
    amax = np.abs(blk).max(axis=-1)
    nz = amax > 0
    _, e2 = np.frexp(np.where(nz, amax, 1.0))
    e = np.clip(e2 - 1 - 8, -127, 127)
    e = np.where(nz, e, 0)
    codes = F.e4m3_encode(blk / np.ldexp(1.0, e)[..., None])
    return codes.reshape(shp).astype(np.uint8), (e + 127).astype(np.uint8)


def split_rows_mxfp8x2(rows_f32: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """The W4A16 mode's device encoding of bf16 activations as two MXFP8
    terms, so that block-scaled FP8 tensor cores can take them.  This is the
    library's own encoding, not a step the pages define: the W4A16 forward
    stays the exact product of the bf16 activations (forward() below), and
    this function exists only to check the device's codes bit for bit.

    Per 32-element block v of a row (K elements):
      hi: Xh = 2^clamp(floor(log2 amax) - 7, -127, 127), codes E4M3_rne(v / Xh);
      lo: r = v - dec(hi) * Xh (exact), Xl = 2^clamp(floor(log2 max|r|) - 7,
          -127, 127), codes E4M3_rne(r / Xl);
    an all-zero block (or residual) gets scale byte 0x7F.  Both quotients
    stay below 256 (their codes at most 256), so no code saturates.  For a bf16 block, dec(hi) * Xh +
    dec(lo) * Xl equals v for every element of magnitude >= 2^(E - 13)
    (E = floor(log2 amax)) and is within 2^(E - 21) of v for the rest.

    Returns codes uint8 [..., 2K] (hi blocks in columns [0, K), lo blocks in
    [K, 2K)) and scale bytes uint8 [..., 2K/32] in the same order."""
    v = np.asarray(rows_f32, dtype=np.float32).astype(np.float64)
    shp = v.shape
    blk = v.reshape(shp[:-1] + (shp[-1] // 32, 32))

    def term(b):
        amax = np.abs(b).max(axis=-1)
        nz = amax > 0
        _, e2 = np.frexp(np.where(nz, amax, 1.0))
        e = np.where(nz, np.clip(e2 - 1 - 7, -127, 127), 0)
        scale = np.ldexp(1.0, e)[..., None]
        codes = F.e4m3_encode(b / scale)
        return codes, (e + 127).astype(np.uint8), F.e4m3_decode(codes) * scale

    hc, hs, hval = term(blk)
    lc, ls, _ = term(blk - hval)
    codes = np.concatenate([hc.reshape(shp), lc.reshape(shp)], axis=-1).astype(np.uint8)
    scales = np.concatenate([hs, ls], axis=-1).astype(np.uint8)
    return codes, scales


@dataclass
class Weights:
    """Expert weights in the user layout of the C ABI.

    W4A8 / W4A16: w1 uint8 [E, 2I, H/2] (packed E2M1), w1_sf uint8 [E, 2I, H/32]
    (E8M0), w2 uint8 [E, H, I/2], w2_sf uint8 [E, H, I/32].
    W8A8: w1 uint8 [E, 2I, H] (E4M3), w2 uint8 [E, H, I] with the same scales.
    Rows 0..I-1 of w1 are the gate projection, rows I..2I-1 the up projection.
    """
    w1: np.ndarray
    w1_sf: np.ndarray
    w2: np.ndarray
    w2_sf: np.ndarray
    mode: int = QUANT_W4A8

    def dense(self, which: int, e: int) -> np.ndarray:
        """float64 [N, K] matrix of expert e's w1 (which=1) or w2 (which=2),
        decoded afresh on each call (each forward decodes an expert once)."""
        w, sf = (self.w1, self.w1_sf) if which == 1 else (self.w2, self.w2_sf)
        if self.mode == QUANT_W8A8:
            return F.mxfp8_dequant(w[e], sf[e])
        return F.mxfp4_dequant(w[e], sf[e])


@dataclass
class Forward:
    routing: Routing
    xq: np.ndarray | None       # uint8 [R, H] FP8 codes (W4A8) / [R, H] (W8A8)
    x_scale: np.ndarray | None  # float32 [R] (W4A8) or uint8 [R, H/32] (W8A8)
    g: np.ndarray               # float32 [R, 2I] GEMM1 output after token scale
    h: np.ndarray               # float32 [R, I] SwiGLU output, bf16-rounded
    hq: np.ndarray | None
    h_scale: np.ndarray | None
    y: np.ndarray               # float32 [R, H]
    out: np.ndarray             # float32 [T, H] bf16-rounded output values


def _exact_dot_f32(a: np.ndarray, b_t: np.ndarray) -> np.ndarray:
    """fl32 of the exact product a @ b_t.T (float64 is exact here)."""
    return (a @ b_t.T).astype(np.float32)


def silu_f32(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)) in float32 [P4793 walkthrough: SwiGLU]."""
    z = z.astype(np.float32)
    with np.errstate(over="ignore"):
        return (z / (np.float32(1.0) + np.exp(-z))).astype(np.float32)


def swiglu_bf16(g: np.ndarray) -> np.ndarray:
    """Step 5: h = silu(gate) * up in float32, rounded to bf16, with gate =
    columns 0..I-1 and up = columns I..2I-1 of the GEMM1 output [P4793
    walkthrough: SwiGLU; P3738 review comments: activation between the
    GEMMs].  Gate-first is this build's reading; the pages fix no order."""
    I = g.shape[1] // 2
    gate, up = g[:, :I], g[:, I:]
    return F.bf16_round((silu_f32(gate) * up).astype(np.float32))


def apply_row_scale(acc: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Per-token scale applied to the float32 accumulator rows [P3738
    Implementation Notes: the activation token scale is applied in the
    epilogue]."""
    return (acc * scale[:, None]).astype(np.float32)


def combine(w: np.ndarray, y: np.ndarray, row_of: np.ndarray) -> np.ndarray:
    """Step 8: out[t] = sum_j w[t, j] * y[row_of[t, j]] (float64 sum in slot
    order), rounded to float32 and then to bf16 [P4793 walkthrough: grouped
    GEMM with finalize fusion -- the top-k-weighted un-permute]."""
    out = np.zeros((row_of.shape[0], y.shape[1]), dtype=np.float64)
    for j in range(row_of.shape[1]):
        out += w[:, j:j + 1].astype(np.float64) * y[row_of[:, j]].astype(np.float64)
    return F.bf16_round(out.astype(np.float32))


def forward(x_bf16_bits: np.ndarray, logits: np.ndarray, weights: Weights,
            top_k: int, mode: int = QUANT_W4A8,
            tokens: np.ndarray | None = None) -> Forward:
    """Steps 1-8 for all tokens, or for the subset ``tokens`` (the output of a
    token depends only on its own x and logits, so a subset is exact).

    ``x_bf16_bits``: uint16 [T, H] raw bf16 activations; ``logits``: float32
    [T, E].  Returns every intermediate; ``out`` holds float32 values that
    are exactly bf16 numbers."""
    x_all = F.bf16_bits_to_f32(x_bf16_bits)
    logits = np.asarray(logits, dtype=np.float32)
    if tokens is not None:
        tokens = np.asarray(tokens, dtype=np.int64)
        x_all = x_all[tokens]
        logits = logits[tokens]
    T, H = x_all.shape
    E = logits.shape[1]
    ids, w = route(logits, top_k)
    rt = expand(ids, w, E)
    R = int(rt.offsets[-1])
    xr = x_all[rt.token_of_row]                         # [R, H] float32
    if mode == QUANT_W4A8:
        # per-token quantisation is the same for each copy of the token
        tq, ts = quantize_rows_fp8(x_all)
        xq = tq[rt.token_of_row]
        xs = ts[rt.token_of_row]
        a1 = F.e4m3_decode(xq)
    elif mode == QUANT_W8A8:
        tq, ts = quantize_rows_mxfp8(x_all)
        xq = tq[rt.token_of_row]
        xs = ts[rt.token_of_row]
        a1 = F.mxfp8_dequant(xq, xs)
    else:
        xq, xs = None, None
        a1 = xr.astype(np.float64)
    I2 = weights.w1.shape[1]
    g = np.zeros((R, I2), dtype=np.float32)
    for e in range(E):
        r0, r1 = int(rt.offsets[e]), int(rt.offsets[e + 1])
        if r1 == r0:
            continue                                   # empty expert: no work
        acc = _exact_dot_f32(a1[r0:r1], weights.dense(1, e))
        if mode == QUANT_W4A8:
            acc = apply_row_scale(acc, xs[r0:r1])
        g[r0:r1] = acc
    h = swiglu_bf16(g)
    if mode == QUANT_W4A8:
        hq, hs = quantize_rows_fp8(h)
        a2 = F.e4m3_decode(hq)
    elif mode == QUANT_W8A8:
        hq, hs = quantize_rows_mxfp8(h)
        a2 = F.mxfp8_dequant(hq, hs)
    else:
        hq, hs = None, None
        a2 = h.astype(np.float64)
    y = np.zeros((R, H), dtype=np.float32)
    for e in range(E):
        r0, r1 = int(rt.offsets[e]), int(rt.offsets[e + 1])
        if r1 == r0:
            continue
        acc = _exact_dot_f32(a2[r0:r1], weights.dense(2, e))
        if mode == QUANT_W4A8:
            acc = apply_row_scale(acc, hs[r0:r1])
        y[r0:r1] = acc
    out = combine(w, y, rt.row_of)
    return Forward(routing=rt, xq=xq, x_scale=xs, g=g, h=h, hq=hq, h_scale=hs,
                   y=y, out=out)


def route_and_quantize(x_bf16_bits: np.ndarray, logits: np.ndarray,
                       top_k: int) -> tuple[Routing, np.ndarray, np.ndarray]:
    """Steps 1-3 only, for every token (used where the GEMM steps are too
    slow to run in full): routing, expansion, and the per-token FP8 codes and
    scales of each expanded row."""
    x = F.bf16_bits_to_f32(x_bf16_bits)
    ids, w = route(np.asarray(logits, np.float32), top_k)
    rt = expand(ids, w, logits.shape[1])
    tq, ts = quantize_rows_fp8(x)
    return rt, tq, ts
