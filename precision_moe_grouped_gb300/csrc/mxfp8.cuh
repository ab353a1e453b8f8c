// mxfp8.cuh -- the OCP MX v1.0 MXFP8 (E4M3 + E8M0) conversion of one
// 32-element block, shared by the activation and h quantisers of the W8A8
// mode.
//
// Pages cited (title and section):
//   [P3614] flashinfer PR #3614, "fix: make the cutlass MoE gemm profiler
//           MXFP8-aware": description and discussion (MXFP8 x MXFP8 MoE GEMMs:
//           E4M3 operands with E8M0 block scales; biased exponent 0x7F = 1.0).
// The conversion rule (shared scale X = 2^(floor(log2 amax) - emax_elem),
// emax of E4M3 = 8, elements rounded to nearest even with saturation) is the
// OCP Microscaling Formats v1.0 specification's.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace moe {

// floor(log2(a)) of a finite a > 0, normal or subnormal (from the bits).
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t u = __float_as_uint(a);
  const int be = static_cast<int>((u >> 23) & 0xFFu);
  return be != 0 ? be - 127 : (31 - __clz(static_cast<int>(u & 0x7FFFFFu))) - 149;
}

// Quantises 32 bf16 values (q[0..3], 16 bytes each, in K order): scale byte
// e + 127 with e = clamp(floor(log2 amax) - 8, -127, 127) (byte 127 for an
// all-zero block), codes = E4M3_rne_satfinite(v * 2^-e) -- the product is
// exact, so the conversion is the only rounding.
__device__ __forceinline__ void mx_quant_block(const uint4 (&q)[4], uint8_t* sbyte,
                                               uint4 (&codes)[2]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(q);
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 f = __bfloat1622float2(b[j]);
    amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  int e = 0;
  if (amax > 0.f) e = max(-127, min(127, floor_log2(amax) - 8));
  *sbyte = static_cast<uint8_t>(e + 127);
  // 2^-e with -e in [-119, 127]: a normal float built from its exponent bits
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 f0 = __bfloat1622float2(b[2 * j]);
    const float2 f1 = __bfloat1622float2(b[2 * j + 1]);
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(f0.x, inv), __fmul_rn(f0.y, inv)), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(f1.x, inv), __fmul_rn(f1.y, inv)), __NV_SATFINITE, __NV_E4M3);
    w[j] = (lo & 0xFFFFu) | (hi << 16);
  }
  codes[0] = make_uint4(w[0], w[1], w[2], w[3]);
  codes[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

}  // namespace moe
