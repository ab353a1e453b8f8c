// mxfp8.cuh -- the OCP MX v1.0 MXFP8 (E4M3 + E8M0) conversion of one
// 32-element block, shared by the activation and h quantisers of the W8A8
// mode, and the two-term MXFP8 split of a bf16 block that carries the W4A16
// mode's activations into the block-scaled FP8 MMA.
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
#include <cuda_fp16.h>
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

// 2^e as a float for e in [-149, 127] (normal or subnormal, exact).
__device__ __forceinline__ float exp2i(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(127 + e) << 23)
                   : __uint_as_float(1u << (e + 149));
}

// One MXFP8 term of 32 exact float values v with emax 7: scale byte e + 127,
// e = clamp(floor(log2 amax) - 7, -127, 127) (byte 127 when all are zero),
// codes E4M3_rne(v * 2^-e).  |v| * 2^-e < 256, so nothing saturates; the
// scaling is exact (a power of two; a product below 2^-126 rounds to a zero
// code either way), so the conversion is the only rounding.  dec receives
// each code's value times 2^e (exact).
__device__ __forceinline__ void mx_term7(const float (&v)[32], uint8_t* sbyte, uint4 (&codes)[2],
                                         float (&dec)[32]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const int e = amax > 0.f ? max(-127, min(127, floor_log2(amax) - 7)) : 0;
  *sbyte = static_cast<uint8_t>(e + 127);
  const float inv = exp2i(-e), sc = exp2i(e);
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(v[4 * j], inv), __fmul_rn(v[4 * j + 1], inv)), __NV_SATFINITE,
        __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(v[4 * j + 2], inv), __fmul_rn(v[4 * j + 3], inv)), __NV_SATFINITE,
        __NV_E4M3);
    w[j] = (lo & 0xFFFFu) | (hi << 16);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const __half_raw hr =
          __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>((w[j] >> (8 * p)) & 0xFFu),
                                  __NV_E4M3);
      dec[4 * j + p] = __fmul_rn(__half2float(__half(hr)), sc);
    }
  }
  codes[0] = make_uint4(w[0], w[1], w[2], w[3]);
  codes[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// One MXFP8 term of a 32-element block spread over an aligned group of 8
// lanes, 4 consecutive elements v[0..3] per lane (call it from all 32 lanes
// of a warp; the four groups hold four blocks): e = clamp(floor(log2 amax) -
// emax, -127, 127) over the block (0 when all are zero); returns the lane's
// four codes E4M3_rne_satfinite(v * 2^-e) (element i in byte i), with the
// scale byte e + 127 in *sbyte and each code's value times 2^e in dec.
// Element for element the arithmetic of mx_quant_block (emax 8) and
// mx_term7 (emax 7).
__device__ __forceinline__ uint32_t mx_quad_term(const float (&v)[4], int emax, uint8_t* sbyte,
                                                 float (&dec)[4]) {
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const int e = amax > 0.f ? max(-127, min(127, floor_log2(amax) - emax)) : 0;
  *sbyte = static_cast<uint8_t>(e + 127);
  const float inv = exp2i(-e), sc = exp2i(e);
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(
      make_float2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(
      make_float2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)), __NV_SATFINITE, __NV_E4M3);
  const uint32_t codes = (lo & 0xFFFFu) | (hi << 16);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const __half_raw hr =
        __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>((codes >> (8 * p)) & 0xFFu),
                                __NV_E4M3);
    dec[p] = __fmul_rn(__half2float(__half(hr)), sc);
  }
  return codes;
}

// The two-term split of 32 bf16 values (q[0..3], in K order): hi = the
// MXFP8 term of the values, lo = the MXFP8 term of the residuals v -
// dec(hi) (exact in float: both lie on the value's bf16 grid or finer).
// dec(hi) + dec(lo) equals v for every element of magnitude >= 2^(E - 13),
// E = floor(log2 amax), and lies within 2^(E - 21) of it otherwise.
__device__ __forceinline__ void split_block(const uint4 (&q)[4], uint8_t* hbyte,
                                            uint4 (&hcodes)[2], uint8_t* lbyte,
                                            uint4 (&lcodes)[2]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(q);
  float v[32], d[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 f = __bfloat1622float2(b[j]);
    v[2 * j] = f.x;
    v[2 * j + 1] = f.y;
  }
  mx_term7(v, hbyte, hcodes, d);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __fsub_rn(v[j], d[j]);
  mx_term7(v, lbyte, lcodes, d);
}

}  // namespace moe
