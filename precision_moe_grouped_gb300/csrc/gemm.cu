// gemm.cu -- persistent, warp-specialised grouped GEMM on the sm_103a tensor
// cores (tcgen05 block-scaled MMA, TMEM accumulators, TMA operand staging).
//
// Pages cited (title and section):
//   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
//           MXFP4xFP8 CUTLASS MoE backend for SM90": Description (MXFP4 weight
//           x FP8 activation grouped GEMM; precomputed work scheduling so the
//           main GEMM loop does no grouped tile lookup; per-token scale
//           epilogue), Implementation Notes (the activation token scale is
//           applied in the epilogue), review comments (64-bit linear work
//           index in the precomputed scheduler; a null TMA descriptor must
//           never reach a kernel).
//   [P4793] flashinfer PR #4793, "Unify MoE CuTe DSL dispatch to be dtype
//           agnostic": walkthrough (grouped GEMM with activation (SwiGLU)
//           fusion).
//
// What differs from the pages' Hopper design: sm_103a has block-scaled MMA,
// so the E8M0 weight scales are applied by the tensor core (staged through
// shared memory into TMEM) instead of being folded into the FP8 operand
// before the MMA, and the FP4 weights are consumed directly by
// .kind::mxf8f6f4 (TMA expands each 16-element group to 16 bytes in shared
// memory).
//
// Orientation ("swap-AB"): the MMA's M = 128 rows are WEIGHT rows (output
// features) and its N columns are TOKENS (expanded rows of one expert), so a
// tile's token count only needs to be a multiple of 16: decode batches of 1-32
// tokens per expert waste no tensor work and prefill tiles hold up to 224.
//   D[m, n] = sum_k W[e, m, k] * Xq[row0 + n, k]     (A = W: E2M1, B = Xq: E4M3)
// Work item = (tile of one expert's rows, 128-row weight M-tile); items are
// handed out statically (item = CTA + i * grid) from the device-built tile
// list, so nothing returns to the host.
//
// Roles (192 threads): warp 0 lane 0 = TMA producer; warp 1 = TMEM owner and
// (lane 0) MMA issuer; warps 2-5 = epilogue (warp w reads TMEM lanes
// 32*(w%4) .. +31).  Two TMEM accumulators let the epilogue of one item
// overlap the main loop of the next.
//
// Epilogues:
//   GEMM1 (SWIGLU): acc * s_x[row] -> h = silu(gate) * up -> bf16 h[row, f].
//     Prepared w1 rows put gate feature f in tile row 32q + i and up feature f
//     in row 32q + i + 16 (i < 16), so a lane pair (i, i+16) of one warp holds
//     gate and up of one feature; one shuffle pairs them.
//   GEMM2: acc * s_h[row] -> bf16 y[row, c].
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

template <int BN, int STAGES>
struct GemmCfg {
  static_assert(BN % 32 == 0 && BN <= 256, "token tile must be a multiple of 32 rows");
  static constexpr int kABytes = kTileM * 128;       // FP4 expanded to 1 byte/element in smem
  static constexpr int kBBytes = BN * 128;           // FP8 tokens x 128 K
  static constexpr int kSFBytes = 512;               // 128 rows x 4 E8M0 bytes
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kABytes;
  static constexpr int kOffSF = kOffB + STAGES * kBBytes;
  static constexpr int kOffSFB = kOffSF + STAGES * kSFBytes;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kOffBar = kOffSFB + 512;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + base alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
  // TMEM columns: two fp32 accumulators of BN columns, 8 columns of constant
  // activation scales (up to 256 tokens), 4 columns of weight scales per stage.
  static constexpr int kColSFB = 2 * BN;
  static constexpr int kColSFA = 2 * BN + 8;
  static constexpr int kColsUsed = 2 * BN + 8 + 4 * STAGES;
  static constexpr int kTmemCols = kColsUsed <= 32    ? 32
                                   : kColsUsed <= 64  ? 64
                                   : kColsUsed <= 128 ? 128
                                   : kColsUsed <= 256 ? 256
                                                      : 512;
  static_assert(kColsUsed <= 512, "TMEM budget exceeded");
};

template <int BN, int STAGES, bool SWIGLU>
__global__ void __launch_bounds__(192, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_x,
                        const uint8_t* __restrict__ w_sf, const int4* __restrict__ tiles,
                        const int32_t* __restrict__ num_tiles_p,
                        const float* __restrict__ row_scale, __nv_bfloat16* __restrict__ out,
                        int m_per_expert, int K, int out_ld, int32_t* __restrict__ status,
                        uint64_t timeout_ns, uint32_t a_tx_bytes) {
  using C = GemmCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MT = m_per_expert / kTileM, KS = K / kTileK;
  const int64_t num_items = static_cast<int64_t>(*num_tiles_p) * MT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  // Activation (B) scales are all 1.0: E8M0 byte 127 everywhere.
  for (int i = threadIdx.x; i < 128; i += blockDim.x)
    reinterpret_cast<uint32_t*>(smem + C::kOffSFB)[i] = 0x7F7F7F7Fu;
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t fills = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
        const int tile = static_cast<int>(item / MT), mt = static_cast<int>(item % MT);
        const int4 td = tiles[tile];
        const int nmma = (td.z + 15) & ~15;
        const int nbox = (nmma + 31) >> 5;
        const uint32_t bytes = a_tx_bytes + static_cast<uint32_t>(nbox) * 4096u + 512u;
        const int wrow = td.x * m_per_expert + mt * kTileM;
        const uint8_t* sf = w_sf + (static_cast<int64_t>(td.x) * MT + mt) * KS * 512;
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(empty + stage, phase ^ 1u, timeout_ns, status, kDevTimeout,
                         abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full + stage, bytes);
          uint8_t* sa = smem + C::kOffA + stage * C::kABytes;
          uint8_t* sb = smem + C::kOffB + stage * C::kBBytes;
          tma_load_2d(sa, &tmap_w, ks * kTileK, wrow, full + stage);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(sb + b * 4096, &tmap_x, ks * kTileK, td.y + 32 * b, full + stage);
          bulk_load(smem + C::kOffSF + stage * C::kSFBytes, sf + static_cast<int64_t>(ks) * 512,
                    512u, full + stage);
          ++fills;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every issued copy must land before the CTA may exit: wait for the
      // last fill of each stage (ignores the abort flag, still bounded).
      int32_t none = 0;
      for (int64_t i = 0; i < STAGES && i < fills; ++i) {
        const int64_t f = fills - 1 - i;
        mbar_wait(full + static_cast<int>(f % STAGES), static_cast<uint32_t>((f / STAGES) & 1),
                  timeout_ns, status, kDevTimeout, &none);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t sfb_desc = smem_desc(smem_u32(smem + C::kOffSFB), 0, 128, 0);
      tc_cp_32x128b_x4(tmem + C::kColSFB, sfb_desc);
      tc_cp_32x128b_x4(tmem + C::kColSFB + 4, sfb_desc);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
        const int4 td = tiles[static_cast<int>(item / MT)];
        const uint32_t nmma = static_cast<uint32_t>((td.z + 15) & ~15);
        if (!mbar_wait(tempty + acc, acc_phase ^ 1u, timeout_ns, status, kDevTimeout,
                       abort_flag))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(full + stage, phase, timeout_ns, status, kDevTimeout, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa = tmem + static_cast<uint32_t>(C::kColSFA + 4 * stage);
          tc_cp_32x128b_x4(sfa, smem_desc(smem_u32(smem + C::kOffSF + stage * C::kSFBytes), 0,
                                          128, 0));
          const uint32_t a0 = smem_u32(smem + C::kOffA + stage * C::kABytes);
          const uint32_t b0 = smem_u32(smem + C::kOffB + stage * C::kBBytes);
#pragma unroll
          for (uint32_t kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = smem_desc(a0 + 32 * kk, 0, 1024, 2);
            const uint64_t bdesc = smem_desc(b0 + 32 * kk, 0, 1024, 2);
            tc_mma_mx(d_tmem, adesc, bdesc, idesc_mx(5, 0, nmma, kk, kk), sfa,
                      tmem + C::kColSFB, (ks > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(empty + stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull + acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // No MMA or TMEM copy may still be running when TMEM is freed.
      tc_commit(drain);
      int32_t none = 0;
      mbar_wait(drain, 0, timeout_ns, status, kDevTimeout, &none);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t item = blockIdx.x; item < num_items; item += gridDim.x) {
      const int tile = static_cast<int>(item / MT), mt = static_cast<int>(item % MT);
      const int4 td = tiles[tile];
      const int row0 = td.y, ntok = td.z, nmma = (td.z + 15) & ~15;
      if (!mbar_wait(tfull + acc, acc_phase, timeout_ns, status, kDevTimeout, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(acc * BN);
      for (int c0 = 0; c0 < nmma; c0 += 16) {
        float v[16];
        tmem_ld_32x32b_x16(tbase + static_cast<uint32_t>(c0), v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = c0 + j;
          v[j] *= n < ntok ? __ldg(row_scale + row0 + n) : 0.f;
        }
        if constexpr (SWIGLU) {
          const bool lo = lane < 16;
          const int f = 64 * mt + 16 * q + (lane & 15);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float send = lo ? v[2 * jj + 1] : v[2 * jj];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            const float g = lo ? v[2 * jj] : recv;
            const float u = lo ? recv : v[2 * jj + 1];
            const float hval = g / (1.0f + expf(-g)) * u;
            const int n = c0 + 2 * jj + (lo ? 0 : 1);
            if (n < ntok)
              out[static_cast<int64_t>(row0 + n) * out_ld + f] = __float2bfloat16_rn(hval);
          }
        } else {
          const int c = mt * kTileM + 32 * q + lane;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = c0 + j;
            if (n < ntok) out[static_cast<int64_t>(row0 + n) * out_ld + c] = __float2bfloat16_rn(v[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty + acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, int STAGES, bool SWIGLU>
cudaError_t launch_variant(const GemmArgs& a, cudaStream_t s) {
  using C = GemmCfg<BN, STAGES>;
  auto kern = grouped_gemm_kernel<BN, STAGES, SWIGLU>;
  static bool attr_set = false;  // per instantiation; set before first launch
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<a.num_sms, 192, C::kSmemBytes, s>>>(
      *a.tmap_w, *a.tmap_x, a.w_sf, a.tiles, a.num_tiles, a.row_scale,
      static_cast<__nv_bfloat16*>(a.out), a.m_per_expert, a.k, a.out_ld, a.status, a.timeout_ns,
      a.a_tx_bytes);
  return cudaGetLastError();
}

}  // namespace

// variant 1: decode tiles (<= 32 tokens, 10-stage weight pipeline);
// variant 2: prefill tiles (<= 224 tokens, 5 stages).
cudaError_t launch_gemm(bool swiglu, int variant, const GemmArgs& a, cudaStream_t s) {
  if (variant == 1) {
    return swiglu ? launch_variant<kDecodeBN, 10, true>(a, s)
                  : launch_variant<kDecodeBN, 10, false>(a, s);
  }
  return swiglu ? launch_variant<kPrefillBN, 5, true>(a, s)
                : launch_variant<kPrefillBN, 5, false>(a, s);
}

}  // namespace moe
