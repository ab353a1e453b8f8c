// gemm_pair.cu -- the grouped GEMM on CTA pairs: one tcgen05 block-scaled
// MMA of M = 256 weight rows (two 128-row M-tiles) spans the two SMs of a
// cluster (.cta_group::2), so each SM stages only half of the token box.
//
// Pages cited (title and section):
//   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
//           MXFP4xFP8 CUTLASS MoE backend for SM90": Description (MXFP4 weight
//           x FP8 activation grouped GEMM with precomputed work scheduling,
//           per-token scale epilogue), Implementation Notes (the activation
//           token scale is applied in the epilogue).
//   [P4793] flashinfer PR #4793, "Unify MoE CuTe DSL dispatch to be dtype
//           agnostic": walkthrough (grouped GEMM with SwiGLU fusion).
//
// Why pairs: on prefill tiles the one-CTA GEMM (gemm.cu) is bound by the
// weight bytes it keeps in flight -- a stage's time is the slot round trip
// (TMA issue -> data -> MMA -> release) over the slots that fit in shared
// memory, and a slot holds a 16 KB expanded weight box plus the tile's whole
// token box (up to 20 KB).  Here the token box is split between the two
// CTAs, so a slot shrinks to 16 + 10 KB and 8 slots fit instead of 6: a
// third more weight bytes in flight per SM, with the same TMEM budget (each
// SM's TMEM holds its own 128 rows of the 256 x N accumulator) and half the
// MMA instructions per SM.
//
// Pair layout (rank r = %cluster_ctarank, r = 0 issues every MMA):
//   work item p of tile t = M-tiles 2p (rank 0) and 2p + 1 (rank 1);
//   A (weights): each CTA stages its own M-tile's 128 x 128 box;
//   B (tokens):  N = tile rows rounded up to 32; rank r stages token rows
//                [row0 + r N/2, row0 + (r+1) N/2) (one box of N/2 rows);
//   scales:      each CTA copies its own weight-scale block into its own
//                TMEM (tcgen05.cp.cta_group::2 issued by rank 0);
//   D:           rank r's TMEM holds rows 128 r .. 128 r + 127 (its M-tile)
//                for all N tokens, read by its own epilogue.
// Barriers: every copy of both CTAs completes on rank 0's full barrier
// (.cta_group::2 TMA); rank 0's MMA commit arrives on the empty and
// accumulator-full barriers of both CTAs (multicast); both epilogues release
// an accumulator buffer on rank 0's tempty barrier (16 arrivals).
// All waits are bounded as in gemm.cu.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

// ------------------------------------------------------ cluster / pair PTX
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of `p`'s counterpart in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// 2-D tiled TMA load into this CTA's shared memory that completes on an
// mbarrier of either CTA of the pair (bar = shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* m, int32_t c0,
                                                 int32_t c1, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}

// TMEM allocation for a CTA pair: one warp of each CTA executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Warp-wide forms (one elected lane issues), issued by rank 0 only.
__device__ __forceinline__ void tc2_cp_32x128b_x4_warp(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(sdesc)
      : "memory");
}

__device__ __forceinline__ void tc2_mma_mx_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t sfa_tmem,
                                                uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Arrive once on the barrier at `bar`'s offset in both CTAs of the pair when
// the issuing thread's earlier tcgen05 operations have completed.
__device__ __forceinline__ void tc2_commit_both_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// ... on this CTA's barrier only.
__device__ __forceinline__ void tc2_commit_local_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Instruction descriptor of the pair MMA: as idesc_mx, with M = 256.
__host__ __device__ constexpr uint32_t idesc_mx_pair(uint32_t a_fmt, uint32_t b_fmt, uint32_t n) {
  return (a_fmt << 7) | (b_fmt << 10) | ((n >> 3) << 17) | (1u << 23) | ((256u >> 4) << 24);
}

template <int BN, int STAGES, int NB>
struct PairCfg {
  static_assert(BN % 32 == 0 && BN / 2 <= kPairBoxRowsAt(kNumXMaps - 1),
                "half a token tile must fit the largest pair box");
  static constexpr int kHalfRows = BN / 2;                     // B rows per CTA, at most
  static constexpr int kProdWarps = 3;
  static constexpr int kStagesPerWarp = (STAGES + kProdWarps - 1) / kProdWarps;
  static_assert(3 * kStagesPerWarp <= 32, "producer lanes must fit a warp");
  static constexpr int kABytes = kTileM * 128;                 // expanded E2M1 box
  static constexpr int kBBytes = kHalfRows * 128;              // E4M3 half token box
  static_assert(kBBytes % 1024 == 0, "B slots must keep the 128-byte swizzle atom aligned");
  static constexpr int kSFBytes = 512;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kABytes;
  static constexpr int kOffSF = kOffB + STAGES * kBBytes;
  static constexpr int kOffSFB = kOffSF + STAGES * kSFBytes;   // constant activation scales
  static constexpr int kNumBars = 2 * STAGES + 2 * NB + 2;
  static constexpr int kOffBar = kOffSFB + 512;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // + base alignment slack + one half box of padding, so that no operand
  // read that starts inside a slot can leave the allocation
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024 + kBBytes;
  static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
  static constexpr int kIssuer = kProdWarps;   // owns TMEM; issues (rank 0)
  static constexpr int kThreads = 32 * (kProdWarps + 1 + kEpiWarps);
  static constexpr int kColSFA = NB * BN;
  static constexpr int kColSFB = kColSFA + 4 * STAGES;
  static constexpr int kColsUsed = kColSFB + 8;
  static constexpr int kTmemCols = kColsUsed <= 256 ? 256 : 512;
  static_assert(kColsUsed <= 512, "TMEM budget exceeded");
};

template <int BN, int STAGES, int NB, bool SWIGLU>
__global__ void __launch_bounds__(PairCfg<BN, STAGES, NB>::kThreads, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ XMaps tmap_xh,
                     const __grid_constant__ CUtensorMap tmap_sf,
                     const int4* __restrict__ tiles, const int32_t* __restrict__ num_tiles_p,
                     const float* __restrict__ row_scale, __nv_bfloat16* __restrict__ out,
                     int m_per_expert, int K, int out_ld, int32_t* __restrict__ status,
                     uint64_t timeout_ns, uint32_t a_tx_bytes) {
  using C = PairCfg<BN, STAGES, NB>;
  extern __shared__ uint8_t smem_raw[];
  // Both CTAs run the same kernel with the same static shared memory, so
  // this aligned base -- and every slot offset below -- is the same in both,
  // which the pair MMA's shared-memory descriptors rely on.
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + NB;
  uint64_t* drain = tempty + NB;   // [0]: MMAs done, [1]: constant scales copied
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cid = static_cast<int>(blockIdx.x >> 1), ncl = static_cast<int>(gridDim.x >> 1);
  const int MT = m_per_expert / kTileM, MTP = MT / 2, KS = K / kTileK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 3);    // rank 0's three producer lanes of the stage
      mbar_init(empty + s, 1);   // the MMA commit
    }
    for (int a = 0; a < NB; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, 2 * kEpiWarps);   // the epilogue warps of both CTAs
    }
    mbar_init(drain, 1);
    mbar_init(drain + 1, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_sf);
    for (int i = 0; i < kNumXMaps; ++i) prefetch_tmap(&tmap_xh.m[i]);
  }
  if (warp == C::kIssuer) tmem_alloc_pair(tmem_slot, C::kTmemCols);
  // W4A8: activation (B) scales are all 1.0 (E8M0 byte 127); the per-token
  // scale is applied in the epilogue.
  for (int i = threadIdx.x; i < 128; i += blockDim.x)
    reinterpret_cast<uint32_t*>(smem + C::kOffSFB)[i] = 0x7F7F7F7Fu;
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers, TMEM and constant block are ready
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (rank == 0 && warp == C::kIssuer) {
    const uint64_t sfb_desc = smem_desc(smem_u32(smem + C::kOffSFB), 0, 128, 0);
    tc2_cp_32x128b_x4_warp(tmem + C::kColSFB, sfb_desc);
    tc2_cp_32x128b_x4_warp(tmem + C::kColSFB + 4, sfb_desc);
    tc2_commit_local_warp(drain + 1);
    int32_t none = 0;
    mbar_wait_warp(drain + 1, 0, timeout_ns, status, kDevTimeout, &none);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  griddep_launch_dependents();
  const WorkLimits lim = work_limits(status);
  const int num_items = checked_num_tiles(num_tiles_p, status, lim) * MTP;
  const uint32_t full0 = cluster_addr(full, 0);   // rank 0's full barriers

  if (warp < C::kProdWarps) {
    // ------------------------------------------------------------ producers
    // As in gemm.cu: stage s in warp s % 3, lanes 3 (s / 3) + {0: weight
    // box, 1: token half box, 2: scale block}.  Both CTAs copy their own
    // share into their own slot; rank 0's lane also announces the bytes of
    // both CTAs on its full barrier, where all the copies complete.
    const int s = warp + C::kProdWarps * (lane / 3), role = lane % 3;
    if (s < STAGES) {
      uint32_t phase = 0;
      bool issued = false;
      // fill f = s + j * STAGES: K stage ks of the pair's it-th item; the
      // counters advance without divisions and the item's tile entry and
      // first weight box are re-read only when the item changes
      int ks = s % KS, item = cid + (s / KS) * ncl;
      int cur_item = -1;
      int4 td = make_int4(0, 0, 0, 0);
      int64_t blk0 = 0;
      int halfn = 16, xm = 0;
      const uint32_t bar = full0 + static_cast<uint32_t>(8 * s);
      while (item < num_items) {
        if (item != cur_item) {
          cur_item = item;
          td = checked_tile(tiles, item / MTP, BN, status, lim);
          const int mt = 2 * (item % MTP) + static_cast<int>(rank);
          blk0 = (static_cast<int64_t>(td.x) * MT + mt) * KS;
          halfn = ((td.z + 31) & ~31) >> 1;   // N / 2, a multiple of 16
          xm = (halfn >> 4) - 1;               // box of exactly N / 2 rows
        }
        const int64_t blk = blk0 + ks;
        if (!mbar_wait(empty + s, phase ^ 1u, timeout_ns, status, kDevTimeout, abort_flag)) break;
        if (role == 0) {
          if (rank == 0) mbar_arrive_expect_tx(full + s, 2u * a_tx_bytes);
          tma_load_2d_pair(smem + C::kOffA + s * C::kABytes, &tmap_w, 0,
                           static_cast<int32_t>(blk * kTileM), bar);
        } else if (role == 1) {
          const uint32_t bx = static_cast<uint32_t>(kPairBoxRowsAt(xm)) * 128u;
          if (rank == 0) mbar_arrive_expect_tx(full + s, 2u * bx);
          tma_load_2d_pair(smem + C::kOffB + s * C::kBBytes, &tmap_xh.m[xm], ks * kTileK,
                           td.y + static_cast<int>(rank) * halfn, bar);
        } else {
          if (rank == 0) mbar_arrive_expect_tx(full + s, 2u * 512u);
          tma_load_2d_pair(smem + C::kOffSF + s * C::kSFBytes, &tmap_sf, 0,
                           static_cast<int32_t>(blk), bar);
        }
        issued = true;
        phase ^= 1u;
        ks += STAGES;
        while (ks >= KS) {
          ks -= KS;
          item += ncl;
        }
      }
      // Rank 0: every issued copy of both CTAs must land before either CTA
      // may exit (bounded, ignores the abort flag).  Rank 1 is held by the
      // final cluster barrier until then.
      if (issued && rank == 0) {
        int32_t none = 0;
        mbar_wait(full + s, phase ^ 1u, timeout_ns, status, kDevTimeout, &none);
      }
    }
  } else if (warp == C::kIssuer) {
    // ------------------------------------------------------------ MMA issuer
    if (rank == 0) {
      const uint64_t adesc0 = smem_desc(smem_u32(smem + C::kOffA), 0, 1024, 2);
      const uint64_t bdesc0 = smem_desc(smem_u32(smem + C::kOffB), 0, 1024, 2);
      const uint64_t sdesc0 = smem_desc(smem_u32(smem + C::kOffSF), 0, 128, 0);
      // Items in order, an item's K stages in order; the inner loop carries
      // only the stage and phase counters (as the one-CTA kernel's single
      // issuer).
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int item = cid, it = 0; ok && item < num_items; item += ncl, ++it) {
        const int4 td = checked_tile(tiles, item / MTP, BN, status, lim);
        const uint32_t nmma = static_cast<uint32_t>((td.z + 31) & ~31);
        const uint32_t id0 = idesc_mx_pair(5, 0, nmma);   // A = E2M1 weights, B = E4M3 tokens
        const int acc = it % NB;
        // both epilogues released this buffer (cluster-scope arrivals)
        if (!mbar_wait_warp(tempty + acc, static_cast<uint32_t>((it / NB) & 1) ^ 1u, timeout_ns,
                            status, kDevTimeout, abort_flag))
          break;
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait_warp(full + stage, phase, timeout_ns, status, kDevTimeout, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa = tmem + static_cast<uint32_t>(C::kColSFA + 4 * stage);
          tc2_cp_32x128b_x4_warp(sfa, sdesc0 + static_cast<uint64_t>(stage * (C::kSFBytes >> 4)));
          const uint64_t ad = adesc0 + static_cast<uint64_t>(stage * (C::kABytes >> 4));
          const uint64_t bd = bdesc0 + static_cast<uint64_t>(stage * (C::kBBytes >> 4));
#pragma unroll
          for (uint32_t kk = 0; kk < 4; ++kk)
            tc2_mma_mx_warp(d_tmem, ad + 2 * kk, bd + 2 * kk, id0 | (kk << 4) | (kk << 29), sfa,
                            tmem + C::kColSFB, (ks > 0 || kk > 0) ? 1u : 0u);
          tc2_commit_both_warp(empty + stage);   // both CTAs' slot is free again
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc2_commit_both_warp(tfull + acc);   // both halves of the accumulator are final
      }
      // No MMA or TMEM copy may still be running when TMEM is freed.
      tc2_commit_local_warp(drain);
      int32_t none = 0;
      mbar_wait_warp(drain, 0, timeout_ns, status, kDevTimeout, &none);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const EpiSched sch{cid, ncl, MTP, 2, static_cast<int>(rank), cluster_addr(tempty, 0)};
    epilogue_loop<BN, 1, NB, SWIGLU>(C::kIssuer + 1, 1, tiles, num_items, sch, tfull, tempty,
                                     tmem, row_scale, out, out_ld, timeout_ns, status,
                                     abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  // Neither CTA leaves (or frees TMEM) while the other may still write into
  // its shared memory or TMEM: rank 0 has drained its MMAs and every copy of
  // both CTAs before it arrives here.
  cluster_sync_all();
  if (warp == C::kIssuer) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

template <int BN, int STAGES, int NB, bool SWIGLU>
cudaError_t launch_pair(const GemmArgs& a, cudaStream_t s) {
  using C = PairCfg<BN, STAGES, NB>;
  auto kern = pair_gemm_kernel<BN, STAGES, NB, SWIGLU>;
  // per instantiation and device: resident clusters, queried before the first launch
  static DeviceOnce max_clusters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.num_sms & ~1));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e;
  std::atomic<int>* mc = device_entry(max_clusters, &e);
  if (!mc) return e;
  int n = mc->load(std::memory_order_acquire);
  if (n == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t q = cfg;
    q.attrs = attr + 1;   // the cluster shape alone
    q.numAttrs = 1;
    if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &q)) != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    mc->store(n, std::memory_order_release);
  }
  // persistent: no more pairs than can be resident at once
  if (static_cast<int>(cfg.gridDim.x / 2) > n) cfg.gridDim = dim3(static_cast<unsigned>(2 * n));
  XMaps xm;
  for (int i = 0; i < kNumXMaps; ++i) xm.m[i] = a.tmap_x_pair[i];
  return cudaLaunchKernelEx(&cfg, kern, *a.tmap_w, xm, *a.tmap_sf, a.tiles, a.num_tiles,
                            a.row_scale, static_cast<__nv_bfloat16*>(a.out), a.m_per_expert, a.k,
                            a.out_ld, a.status, a.timeout_ns, a.a_tx_bytes);
}

}  // namespace

bool gemm_pair_supported(int m_per_expert, int act) {
  return act == kActFp8Row && m_per_expert % (2 * kTileM) == 0;
}

cudaError_t launch_gemm_pair(bool swiglu, const GemmArgs& a, cudaStream_t s) {
  if (!gemm_pair_supported(a.m_per_expert, a.act) || a.num_sms < 2 || !a.tmap_x_pair)
    return cudaErrorInvalidValue;
  return swiglu ? launch_pair<kPairBN, kPairStages, 2, true>(a, s)
                : launch_pair<kPairBN, kPairStages, 2, false>(a, s);
}

}  // namespace moe
