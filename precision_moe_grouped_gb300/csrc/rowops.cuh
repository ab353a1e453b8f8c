// rowops.cuh -- the per-row arithmetic of the h quantisation (its kernels
// are in rowops.cu).
//
// Pages cited (title and section):
//   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
//           MXFP4xFP8 CUTLASS MoE backend for SM90": Description (per-token FP8
//           scales threaded through activation and GEMM1/GEMM2), review
//           comments (FP8 x MXFP4 quant params carry fc1 and fc2 token scales).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace moe {

// Per-row FP8 quantisation of h row r (bf16 [R, I]) by one warp: amax,
// s2 = amax/448, codes = E4M3_rne_satfinite(h * (448/amax)) (IEEE
// divisions); an all-zero row gets s2 = 1 and zero codes.  Lane l keeps the
// 16-element vectors l, l + 32, ... of the row (up to 4 of them, I <= 2048)
// in registers between the amax pass and the conversion; longer rows are
// read again for the conversion.  Rows are read through L2 (ld.global.cg):
// each element is read once.
__device__ __forceinline__ void hquant_row_warp(const __nv_bfloat16* __restrict__ h, int r, int I,
                                                uint8_t* __restrict__ hq,
                                                float* __restrict__ h_scale, int lane) {
  constexpr int kKeep = 4;
  const uint4* hr = reinterpret_cast<const uint4*>(h + static_cast<size_t>(r) * I);
  const int nvec = I / 16;
  uint4 keep[kKeep][2];
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < kKeep; ++c) {
    const int i = lane + 32 * c;
    if (i < nvec) {
      keep[c][0] = __ldcg(hr + 2 * i);
      keep[c][1] = __ldcg(hr + 2 * i + 1);
    }
  }
  for (int i = lane; i < nvec; i += 32) {
    uint4 q[2];
    const int c = (i - lane) / 32;
    if (c < kKeep) {
#pragma unroll
      for (int cc = 0; cc < kKeep; ++cc)
        if (cc == c) {
          q[0] = keep[cc][0];
          q[1] = keep[cc][1];
        }
    } else {
      q[0] = __ldcg(hr + 2 * i);
      q[1] = __ldcg(hr + 2 * i + 1);
    }
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(q);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const bool nz = amax > 0.f;
  const float inv = nz ? 448.0f / amax : 0.0f;
  uint4* dst = reinterpret_cast<uint4*>(hq + static_cast<size_t>(r) * I);
  for (int i = lane; i < nvec; i += 32) {
    uint4 out = make_uint4(0, 0, 0, 0);
    if (nz) {
      uint4 q[2];
      const int c = (i - lane) / 32;
      if (c < kKeep) {
#pragma unroll
        for (int cc = 0; cc < kKeep; ++cc)
          if (cc == c) {
            q[0] = keep[cc][0];
            q[1] = keep[cc][1];
          }
      } else {
        q[0] = __ldcg(hr + 2 * i);
        q[1] = __ldcg(hr + 2 * i + 1);
      }
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(q);
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f0 = __bfloat1622float2(b[2 * j]);
        const float2 f1 = __bfloat1622float2(b[2 * j + 1]);
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(f0.x, inv), __fmul_rn(f0.y, inv)), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(f1.x, inv), __fmul_rn(f1.y, inv)), __NV_SATFINITE, __NV_E4M3);
        w[j] = (lo & 0xFFFFu) | (hi << 16);
      }
      out = make_uint4(w[0], w[1], w[2], w[3]);
    }
    dst[i] = out;
  }
  if (lane == 0) h_scale[r] = nz ? amax / 448.0f : 1.0f;
}

// hquant_row_warp on a row already staged in shared memory (hs: I bf16):
// the same arithmetic, both passes reading shared memory.
__device__ __forceinline__ void hquant_row_smem(const __nv_bfloat16* hs, int r, int I,
                                                uint8_t* __restrict__ hq,
                                                float* __restrict__ h_scale, int lane) {
  const uint4* hr = reinterpret_cast<const uint4*>(hs);
  const int nvec = I / 16;
  float amax = 0.f;
  for (int i = lane; i < nvec; i += 32) {
    const uint4 q[2] = {hr[2 * i], hr[2 * i + 1]};
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(q);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const bool nz = amax > 0.f;
  const float inv = nz ? 448.0f / amax : 0.0f;
  uint4* dst = reinterpret_cast<uint4*>(hq + static_cast<size_t>(r) * I);
  for (int i = lane; i < nvec; i += 32) {
    uint4 out = make_uint4(0, 0, 0, 0);
    if (nz) {
      const uint4 q[2] = {hr[2 * i], hr[2 * i + 1]};
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(q);
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f0 = __bfloat1622float2(b[2 * j]);
        const float2 f1 = __bfloat1622float2(b[2 * j + 1]);
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(f0.x, inv), __fmul_rn(f0.y, inv)), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(f1.x, inv), __fmul_rn(f1.y, inv)), __NV_SATFINITE, __NV_E4M3);
        w[j] = (lo & 0xFFFFu) | (hi << 16);
      }
      out = make_uint4(w[0], w[1], w[2], w[3]);
    }
    dst[i] = out;
  }
  if (lane == 0) h_scale[r] = nz ? amax / 448.0f : 1.0f;
}

}  // namespace moe
