"""Writes exact_swiglu_case.json: a hand-derivable fused-MoE case whose every
intermediate is an exact small multiple of a power-of-two-times-49 number.

The pages print no worked example, so this fixture is derived in closed form
(integer arithmetic only; torch is used solely to round the final integers to
bf16).  Structure, for E = 2 experts, H = 64, I = 32:
  x[t]        = 448 at one position p_t (p = 0 for token 0, p = 33 for token 1:
                low nibble of block 0 and high nibble of block 1), 0 elsewhere.
                => amax = 448, s = 1, inv = 1: FP8 codes exact, 0x7E at p.
  w1[e]       gate row n: rho[e][n] * 1 at k=0 and k=33; up row n: sigma[e][n]
                at k=0 and k=33.  Scale byte 127 for block 0, 128 (x2) for
                block 1, so the weight value at k=33 is doubled.
  => token t (scale factor m_t = 1 for t=0, 2 for t=1): gate = 448 m rho,
     up = 448 m sigma.  silu(448 m) = 448 m exactly in float32 (exp(-448m)
     underflows to 0), silu(-448 m) = -0 (exp overflows to inf).
     h_j = (448 m)^2 sigma_j if rho_j = +1 else 0 -- exact in bf16.
  h-quant: amax_h = (448 m)^2 (if any rho = +1), s2 = 448 m^2 exactly and
     every nonzero h code is +-448 (0x7E / 0xFE).  An all-zero h row gets
     s2 = 1 and codes 0.
  w2[e][c][j] = tau[e][c][j] in {0, +-1, +-2}, scale byte 127.
  => y_e[c] = s2 * sum_j (448 sigma_j [rho_j>0]) tau[c][j]
            = (448 m)^2 * S_e[c],  S_e[c] = sum_j [rho_j > 0] sigma_j tau[c][j].
  combine: out[t][c] = bf16(sum_{e in top-k(t)} w_te * y_e[c]), with w = 1
     for k = 1 and w = 1/2 exactly for k = 2 with equal logits.
The same case in the other two quantisation modes:
  W4A16 (bf16 activations, MXFP4 weights, h fed to GEMM2 as bf16): x = 448
     enters unquantised and h = (448 m)^2 sigma_j is exact in bf16
     ((448 m)^2 = 49 * 2^(12 + 2 log2 m)), so y and out equal the W4A8 values.
  W8A8 (MXFP8 x MXFP8, OCP MX blocks of 32): the same weight values as E4M3
     codes (+-1 = 0x38/0xB8, +-2 = 0x40/0xC0) with the same scale bytes.  x's
     block holding 448 has amax 448 = 1.75 * 2^8, so X = 2^(8 - 8) = 1 and the
     code is 0x7E; all-zero blocks get byte 127 and zero codes.  GEMM1 and
     SwiGLU are as above.  The h row (I = 32, one block) has amax (448 m)^2 =
     392 * 2^(9 + 2 log2 m), so X = 2^(9 + 2 log2 m) (scale byte 136 for
     m = 1, 138 for m = 2) and each nonzero h / X = +-392, which E4M3 cannot
     hold: round-to-nearest gives +-384 (code 0x7C / 0xFC; the neighbours are
     384 and 416).  Hence y_e[c] = 384 * X * S_e[c] = 196608 m^2 S_e[c] and
     out[t][c] = bf16(sum w_te * 196608 m^2 S_e[c]).
Run: python tests/golden/make_exact_swiglu_case.py
"""
import json
import os

import numpy as np
import torch

E, H, I = 2, 64, 32


def _bf16(v) -> list:
    """float64 values (exact integers here) rounded to bf16, as floats."""
    return torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).to(torch.float32).tolist()


def main():
    rng = np.random.default_rng(2024)
    rho = rng.choice([1, -1], size=(E, I))
    rho[1, :] = -1          # expert 1: every gate negative -> all-zero h rows
    sigma = rng.choice([1, -1], size=(E, I))
    tau = np.zeros((E, H, I), dtype=np.int64)
    for e in range(E):
        for c in range(H):
            js = rng.choice(I, size=2, replace=False)
            tau[e, c, js] = rng.choice([1, -1, 2, -2], size=2)
    cases = []
    for k, logits in [(1, [[1.0, 0.0], [0.0, 1.0]]), (2, [[0.5, 0.5], [-1.0, -1.0]])]:
        out = np.zeros((2, H), dtype=np.float64)
        out_w8a8 = np.zeros((2, H), dtype=np.float64)
        for t in range(2):
            m = 1 if t == 0 else 2
            chosen = [int(np.argmax(logits[t]))] if k == 1 else [0, 1]
            w = 1.0 if k == 1 else 0.5
            for e in chosen:
                S = ((rho[e] > 0) * sigma[e] * tau[e]).sum(axis=1)   # integer [H]
                out[t] += w * (448 * m) ** 2 * S
                out_w8a8[t] += w * 196608 * m * m * S
        cases.append({"top_k": k, "logits": logits, "expected_out": _bf16(out),
                      "expected_out_w4a16": _bf16(out), "expected_out_w8a8": _bf16(out_w8a8)})
    doc = {
        "source": "closed-form case; derivation in make_exact_swiglu_case.py. Steps follow "
                  "flashinfer PR #3738 'perf: optimize MXFP4xBF16 & INT4xFP8 and add MXFP4xFP8 "
                  "CUTLASS MoE backend for SM90' (Description: runtime per-token FP8 activation "
                  "quantization, MXFP4 weights, per-token scale epilogue) and PR #4793 'Unify MoE "
                  "CuTe DSL dispatch to be dtype agnostic' (SwiGLU activation, finalize).",
        "E": E, "H": H, "I": I, "x_positions": [0, 33], "w1_block_scale_bytes": [127, 128],
        "rho": rho.tolist(), "sigma": sigma.tolist(), "tau": tau.tolist(), "cases": cases,
        "w8a8_h_code_magnitude": 0x7C, "w8a8_h_scale_bytes": [136, 138],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "exact_swiglu_case.json")
    with open(path, "w") as f:
        json.dump(doc, f)


if __name__ == "__main__":
    main()
