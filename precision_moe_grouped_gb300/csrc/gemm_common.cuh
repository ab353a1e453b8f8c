// gemm_common.cuh -- pieces shared by the grouped GEMM kernels (gemm.cu: one
// CTA per tile; gemm_pair.cu: CTA pairs): the activation tensor-map set and
// the TMEM -> registers -> global epilogue.
//
// Pages cited (title and section):
//   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
//           MXFP4xFP8 CUTLASS MoE backend for SM90": Implementation Notes
//           (the activation token scale is applied in the epilogue).
//   [P4793] flashinfer PR #4793, "Unify MoE CuTe DSL dispatch to be dtype
//           agnostic": walkthrough (grouped GEMM with activation (SwiGLU)
//           fusion).
#pragma once

#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

// Activation tensor maps with box heights 16, 32, 64, ..., 224 rows: a tile
// loads the smallest box covering its MMA-N rows in one copy.
struct XMaps {
  CUtensorMap m[kNumXMaps];
};

__device__ __forceinline__ int x_map_for(int rows) {
  return rows <= 16 ? 0 : (rows + 31) / 32;
}

// Number of epilogue warps: two per TMEM lane quarter.
constexpr int kEpiWarps = 8;

// ------------------------------------------------------- checked builds
// The work-map limits a checked build validates against: R expanded rows and
// E experts, recorded by the forward's first kernel (zeros otherwise).
struct WorkLimits {
  int R, E;
};

__device__ __forceinline__ WorkLimits work_limits(const int32_t* status) {
  if constexpr (kChecks) return WorkLimits{status[2], status[3]};
  return WorkLimits{0, 0};
}

// The tile count; a checked build records MOE_ERR_DEVICE_CHECK and runs no
// tiles when it exceeds the largest list the expansion can build.
__device__ __forceinline__ int checked_num_tiles(const int32_t* num_tiles_p, int32_t* status,
                                                 WorkLimits lim) {
  const int n = *num_tiles_p;
  if constexpr (kChecks) {
    if (n < 0 || n > max_work_tiles(lim.R, lim.E, kTinyBN)) {
      atomicCAS(status, 0, kDevCheckFailed);
      return 0;
    }
  }
  return n;
}

// Tile entry i (expert, first row, rows, 0).  A checked build replaces an
// entry out of range (expert >= E, rows outside [0, R), more than bn rows)
// by a harmless 16-row tile of expert 0 marked w = 1, whose outputs the
// epilogue does not store, and records MOE_ERR_DEVICE_CHECK.  Every role of
// a GEMM reads the entry through this function, so all agree.
__device__ __forceinline__ int4 checked_tile(const int4* __restrict__ tiles, int i, int bn,
                                             int32_t* status, WorkLimits lim) {
  int4 td = tiles[i];
  if constexpr (kChecks) {
    if (!tile_entry_ok(td.x, td.y, td.z, td.w, bn, lim.R, lim.E)) {
      atomicCAS(status, 0, kDevCheckFailed);
      td = make_int4(0, 0, 16, 1);
    }
  }
  return td;
}

// The epilogue of a persistent grouped GEMM whose TMEM holds, per
// accumulator buffer a, NI partial accumulators of BN fp32 columns (issuer
// i's at column (a * NI + i) * BN; ni of them in use), row m = weight row
// (output feature) m of the item's 128-row M-tile, column n = the tile's
// n-th token.  Warps first_warp .. first_warp + 7: warp w reads TMEM lanes
// 32 * (w % 4) .. +31 (the only quarter it may access); the two warps of a
// quarter split the item's 16-column chunks.  Each chunk: sum the partials,
// multiply column n by row_scale[row0 + n] (1 when row_scale is null), then
//   SWIGLU: tile rows 32q + i (gate) and 32q + 16 + i (up) of feature
//     64 mt + 16q + i sit in lanes i and i + 16 of one warp; one shuffle
//     pairs them, h = silu(g) * u -> bf16 out[row, feature];
//   else:   bf16 out[row, 128 mt + 32q + lane].
// Releases the accumulator buffer (tempty) after reading it.
//
// EpiSched says which items this CTA's epilogue visits and where their
// weight M-tile is: items item0, item0 + item_step, ...; item -> tile
// item / items_per_tile, M-tile (item % items_per_tile) * mt_mul + mt_add.
// A CTA that runs its own MMAs uses (blockIdx.x, gridDim.x, MT, 1, 0).  In a
// CTA pair the item is an M-tile pair and CTA rank r holds M-tile 2p + r;
// its buffer release goes to the MMA-issuing CTA's tempty barrier, whose
// shared::cluster address is release_cluster (0: the local tempty).
struct EpiSched {
  int item0, item_step, items_per_tile, mt_mul, mt_add;
  uint32_t release_cluster;
};

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Top-k combine formed in GEMM2's epilogue (moe_options.fuse_combine; null
// cnt = off).  After a warp has stored its 32 columns of y for a chunk of
// tokens, it counts, per token t of the chunk, one arrival on
// cnt[(t * MT + mt) * 4 + q] (q = its lane quarter); the warp whose arrival
// is the k-th combines that 32-column segment of t: out[t, c] = bf16(sum over
// slots j in order of fmaf(w[t, j], y[row_of[t, j], c], acc)) -- the combine
// kernel's arithmetic -- and clears the counter.  Release: every lane fences
// its y stores before the arrivals; acquire: a fence before reading the
// other rows (written by other CTAs) through L2.
struct CombineArgs {
  int32_t* cnt;             // [T, MT, 4], zero when the kernel starts
  const int32_t* slot;      // token_slot [R]: token = slot / k
  const int32_t* row_of;    // [T, k]
  const float* wts;         // [T, k]
  __nv_bfloat16* out;       // [T, out_ld]
  int k, MT;
};

// EW = epilogue warps: 8 (two per lane quarter, splitting the chunks) or 4
// (one per quarter).
template <int BN, int NI, int NB, bool SWIGLU, int EW = kEpiWarps>
__device__ __forceinline__ void epilogue_loop(int first_warp, int ni, const int4* __restrict__ tiles,
                                              int num_items, EpiSched sch, uint64_t* tfull,
                                              uint64_t* tempty, uint32_t tmem,
                                              const float* __restrict__ row_scale,
                                              __nv_bfloat16* __restrict__ out, int out_ld,
                                              uint64_t timeout_ns, int32_t* status,
                                              volatile int32_t* abort_flag,
                                              const CombineArgs cmb = CombineArgs{}) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;
  static_assert(EW == 4 || EW == 8, "one or two epilogue warps per TMEM lane quarter");
  const int half = EW == 8 ? (warp - first_warp) >> 2 : 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  const WorkLimits lim = work_limits(status);
  for (int item = sch.item0; item < num_items; item += sch.item_step) {
    const int tile = item / sch.items_per_tile;
    const int mt = (item % sch.items_per_tile) * sch.mt_mul + sch.mt_add;
    const int4 td = checked_tile(tiles, tile, BN, status, lim);
    const int row0 = td.y, ntok = (kChecks && td.w) ? 0 : td.z;   // a replaced tile stores nothing
    const int nchunks = (ntok + 15) >> 4;
    const int split = EW == 8 ? (nchunks + 1) >> 1 : nchunks;
    const int ch_begin = half == 0 ? 0 : split, ch_end = half == 0 ? split : nchunks;
    if (!mbar_wait(tfull + acc, acc_phase, timeout_ns, status, kDevTimeout, abort_flag)) break;
    tc_fence_after();
    const uint32_t tbase =
        tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(acc * NI * BN);
    for (int ch = ch_begin; ch < ch_end; ++ch) {
      const int c0 = ch * 16;
      // one row-scale load per chunk: lane j (and j + 16) holds column c0 + j
      const int nl = c0 + (lane & 15);
      const float sc = nl < ntok ? (row_scale ? __ldg(row_scale + row0 + nl) : 1.f) : 0.f;
      float v[16];
      tmem_ld_32x32b_x16(tbase + static_cast<uint32_t>(c0), v);
      for (int p = 1; p < ni; ++p) {   // partial sums of the other issuers
        float w[16];
        tmem_ld_32x32b_x16(tbase + static_cast<uint32_t>(p * BN + c0), w);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] += w[j];
      }
      if constexpr (SWIGLU) {
        // After the exchange a lane holds gate and up of one (feature, token)
        // pair, so the token's scale is applied to those two values only.
        const bool lo = lane < 16;
        const int f = 64 * mt + 16 * q + (lane & 15);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float send = lo ? v[2 * jj + 1] : v[2 * jj];
          const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
          const float s_n = __shfl_sync(0xffffffffu, sc, 2 * jj + (lo ? 0 : 1));
          const float g = (lo ? v[2 * jj] : recv) * s_n;
          const float u = (lo ? recv : v[2 * jj + 1]) * s_n;
          // silu(g) = g / (1 + e^-g); fast exp and division (relative error
          // ~1e-6, far below the bf16 rounding of h that follows)
          const float hval = __fdividef(g, 1.0f + __expf(-g)) * u;
          const int n = c0 + 2 * jj + (lo ? 0 : 1);
          if (n < ntok)
            out[static_cast<int64_t>(row0 + n) * out_ld + f] = __float2bfloat16_rn(hval);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] *= __shfl_sync(0xffffffffu, sc, j);
        const int c = mt * kTileM + 32 * q + lane;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = c0 + j;
          if (n < ntok) out[static_cast<int64_t>(row0 + n) * out_ld + c] = __float2bfloat16_rn(v[j]);
        }
        if (cmb.cnt) {
          __threadfence();
          __syncwarp();
          int tt = 0;
          bool last = false;
          if (lane < 16 && c0 + lane < ntok) {
            tt = __ldg(cmb.slot + row0 + c0 + lane) / cmb.k;
            last = atomicAdd(cmb.cnt + (static_cast<int64_t>(tt) * cmb.MT + mt) * 4 + q, 1) ==
                   cmb.k - 1;
          }
          unsigned pend = __ballot_sync(0xffffffffu, last);
          if (pend) __threadfence();
          while (pend) {
            const int src = __ffs(pend) - 1;
            pend &= pend - 1;
            const int t = __shfl_sync(0xffffffffu, tt, src);
            const int64_t tk = static_cast<int64_t>(t) * cmb.k;
            float acc = 0.f;
            for (int j = 0; j < cmb.k; ++j) {
              const int64_t r = __ldg(cmb.row_of + tk + j);
              const unsigned short yb =
                  __ldcg(reinterpret_cast<const unsigned short*>(out + r * out_ld + c));
              acc = fmaf(__ldg(cmb.wts + tk + j), __bfloat162float(__ushort_as_bfloat16(yb)), acc);
            }
            cmb.out[static_cast<int64_t>(t) * out_ld + c] = __float2bfloat16_rn(acc);
            if (lane == 0) cmb.cnt[(static_cast<int64_t>(t) * cmb.MT + mt) * 4 + q] = 0;
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (sch.release_cluster)
        mbar_arrive_cluster(sch.release_cluster + static_cast<uint32_t>(8 * acc));
      else
        mbar_arrive(tempty + acc);
    }
    if (++acc == NB) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
}

}  // namespace moe
