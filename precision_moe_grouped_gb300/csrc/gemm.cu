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
// Operands by activation encoding (ACT): W4A8 -- A = E2M1 weights, B = E4M3
// activations with constant unit block scales (the per-row token scale is
// applied in the epilogue); W8A8 -- A = E4M3 weights, B = E4M3 activations
// with their per-32 block scales; W4A16 -- A = E2M1 weights and B = the two
// MXFP8 terms of the bf16 activations (hi, lo): each stage holds both terms'
// boxes and scale blocks, and its MMAs accumulate A x hi and A x lo into
// one accumulator, so the bf16 product runs on the FP8 tensor pipe.
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
// Roles: the first warps = TMA producers (one warp per pipeline stage, three
// lanes per stage); the next NI warps = MMA issuers (one elected lane each;
// the first also owns the TMEM allocation); the next 8 warps = epilogue
// (warp w reads TMEM lanes 32*(w%4) .. +31; two warps per lane quarter split
// the columns); the last warp = optional L2 prefetcher.  Two TMEM accumulator
// buffers let the epilogue of one item overlap the main loop of the next.
//
// Gathered activations (W4A8 GEMM1, opt-in): with gather_slot set, the
// activations are token-major ([T, K]: each token's FP8 row written once by
// the expansion) and each stage's producer warp copies the tile's rows by
// token (token = gather_slot[row] / gather_k) with 16-byte asynchronous
// copies into the slot's 128-byte-swizzled box, arriving on the slot's
// barrier as they land -- the gather-fused grouped GEMM of [P4793] (file
// list: blockscaled_contiguous_gather_grouped_gemm_act_fusion), without the
// expanded [R, K] copy.
//
// Epilogues:
//   GEMM1 (SWIGLU): acc * s_x[row] -> h = silu(gate) * up -> bf16 h[row, f].
//     Prepared w1 rows put gate feature f in tile row 32q + i and up feature f
//     in row 32q + i + 16 (i < 16), so a lane pair (i, i+16) of one warp holds
//     gate and up of one feature; one shuffle pairs them.
//   GEMM2: acc * s_h[row] -> bf16 y[row, c].
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

template <int BN, int STAGES, int NI, int NB, int ACT>
struct GemmCfg {
  static_assert(BN % 16 == 0 && BN <= kXBoxRowsAt(kNumXMaps - 1),
                "token tile must be a multiple of 16 rows and fit the largest box");
  static constexpr bool kTiledSfb = ACT != kActFp8Row;   // per-tile activation scales
  static constexpr bool kSplit = ACT == kActSplit;       // two activation terms per stage
  static_assert(!kSplit || BN <= 128, "a split stage holds one 512-byte scale block per term");
  // Producer warps: stage s is served by warp s % kProdWarps, with three
  // lanes per stage (weight, activation and scale copies), or two (the scale
  // copy rides with the activation) if three do not fit a warp.  Lanes of one
  // warp waiting on different stages' barriers serialise, so each stage gets
  // its own warp (against three warps sharing the stages: DSV3 T=1 54.5 ->
  // 51.9 us, T=512 981 -> 941 us, T=4096 1566 -> 1548 us, W4A16 T=256 77.4
  // -> 73.3 us; MXFP8 Zipf T=4096 2021 -> 1965 us once the issuer elects
  // once per stage).
  static constexpr int kProdWarps = STAGES;
  static constexpr int kStagesPerWarp = (STAGES + kProdWarps - 1) / kProdWarps;
  static constexpr int kLanesPerStage = 3 * kStagesPerWarp <= 32 ? 3 : 2;
  static_assert(kLanesPerStage * kStagesPerWarp <= 32, "producer lanes must fit a warp");
  static_assert(STAGES % NI == 0, "each stage must belong to one MMA issuer");
  static constexpr int kABytes = kTileM * 128;       // FP4 expanded to 1 byte/element in smem
  static constexpr int kTermBytes = BN * 128;        // FP8 tokens x 128 K
  static constexpr int kBBytes = (kSplit ? 2 : 1) * kTermBytes;
  static constexpr int kSFBytes = 512;               // 128 rows x 4 E8M0 bytes
  // MXFP8 / split: the activation scales of a stage, 512 bytes per 128 tile
  // rows (per term)
  static constexpr int kSFBSlot = kTiledSfb ? 512 * ((BN + 127) / 128) * (kSplit ? 2 : 1) : 0;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kABytes;
  static constexpr int kOffSF = kOffB + STAGES * kBBytes;
  static constexpr int kOffSFBs = kOffSF + STAGES * kSFBytes;
  static constexpr int kOffSFB = kOffSFBs + STAGES * kSFBSlot;   // constant scales (W4A8)
  static constexpr int kNumBars = 2 * STAGES + 2 * NB + 1 + NI;
  static constexpr int kOffBar = kOffSFB + (kTiledSfb ? 0 : 512);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // W4A8: each producer warp's token list of its current tile (one int per
  // tile row) for GEMM1 gathering token-major activations, where it fits
  static constexpr int kTokBytes = ACT == kActFp8Row ? kProdWarps * BN * 4 : 0;
  static constexpr bool kGatherFits =
      kTokBytes > 0 && kOffMisc + 16 + kTokBytes + 1024 <= 232448;
  static constexpr int kOffTok = kOffMisc + 16;
  static constexpr int kSmemBytes =
      kOffMisc + 16 + (kGatherFits ? kTokBytes : 0) + 1024;   // + base alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
  // TMEM columns: for each of the NB accumulator buffers, one fp32
  // accumulator of BN columns per MMA issuer (buffer a, issuer i at column
  // (a * NI + i) * BN); 4 columns of weight scales per stage; activation
  // scales: 8 columns of constants (W4A8, up to 256 tokens) or 8 columns per
  // stage (MXFP8: rows 0-127 and 128-255; split: the hi and the lo term).
  // producer, issuers, epilogue, L2 prefetcher
  static constexpr int kIssuer0 = kProdWarps;   // first issuer warp; owns TMEM
  static constexpr int kThreads = 32 * (kProdWarps + NI + kEpiWarps + 1);
  static constexpr int kColSFA = NB * NI * BN;
  static constexpr int kColSFB = kColSFA + 4 * STAGES;
  static constexpr int kColsUsed = kColSFB + (kTiledSfb ? 8 * STAGES : 8);
  static constexpr int kTmemCols = kColsUsed <= 32    ? 32
                                   : kColsUsed <= 64  ? 64
                                   : kColsUsed <= 128 ? 128
                                   : kColsUsed <= 256 ? 256
                                                      : 512;
  static_assert(kColsUsed <= 512, "TMEM budget exceeded");
};

template <int BN, int STAGES, int NI, int NB, bool SWIGLU, int ACT>
__global__ void __launch_bounds__(GemmCfg<BN, STAGES, NI, NB, ACT>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ XMaps tmap_x,
                        const __grid_constant__ CUtensorMap tmap_sf,
                        const int4* __restrict__ tiles,
                        const int32_t* __restrict__ num_tiles_p,
                        const float* __restrict__ row_scale, __nv_bfloat16* __restrict__ out,
                        int m_per_expert, int K, int out_ld, int32_t* __restrict__ status,
                        uint64_t timeout_ns, uint32_t a_tx_bytes, int prefetch_stages,
                        const uint8_t* __restrict__ sfb_tiled,
                        const uint8_t* __restrict__ w_base, int max_tiles, int early_list,
                        const int32_t* __restrict__ gather_slot, int gather_k,
                        const uint8_t* __restrict__ xg, const CombineArgs cmb) {
  using C = GemmCfg<BN, STAGES, NI, NB, ACT>;
  // A = E2M1 weights, or E4M3 in MXFP8; B = activations: E4M3
  constexpr uint32_t kAFmt = ACT == kActMxfp8 ? 0u : 5u;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + NB;
  uint64_t* drain = tempty + NB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + C::kOffMisc + 4);
  // last fill whose MMAs the first issuer has issued (paces the prefetcher)
  volatile int32_t* progress = reinterpret_cast<volatile int32_t*>(smem + C::kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MT = m_per_expert / kTileM, KS = K / kTileK;
  // Issuers with work: the largest divisor of STAGES that is <= min(NI, KS).
  // Dividing STAGES makes every stage always consumed by the same issuer
  // (fill f -> stage f % STAGES -> issuer f % ni), so each full barrier is
  // waited on in phase order by one thread; a second thread waiting on the
  // same barrier could see the parity of an older phase and run ahead.
  // ni <= KS gives every issuer at least one stage of every item.
  int ni = NI < KS ? NI : KS;
  while (STAGES % ni != 0) --ni;

  // GEMM1 of W4A8 with gather_slot: the activations are token-major (xg,
  // [T, K] codes); each stage's producer warp copies the weights and scales
  // (lane 0, one arrival) and gathers the tile's rows by token with vector
  // loads and swizzled shared stores (one more arrival).
  const bool gather = C::kGatherFits && ACT == kActFp8Row && SWIGLU && gather_slot != nullptr;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // each producer lane arrives with its bytes (gathering: lane 0 with
      // the weight bytes, and every lane of the warp once its copies land)
      mbar_init(full + s, gather ? 1 + 32 : C::kLanesPerStage);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < NB; ++a) {
      mbar_init(tfull + a, ni);   // every issuer commits its share of an item
      mbar_init(tempty + a, kEpiWarps);   // every epilogue warp releases the buffer
    }
    for (int j = 0; j < NI; ++j) mbar_init(drain + j, 1);
    mbar_init(drain + NI, 1);   // constant-scale copy done
    *abort_flag = 0;
    *progress = -1;
    fence_mbar_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_sf);
    for (int i = 0; i < kNumXMaps; ++i) prefetch_tmap(&tmap_x.m[i]);
  }
  if (warp == C::kIssuer0) tmem_alloc(tmem_slot, C::kTmemCols);
  // W4A8: activation (B) scales are all 1.0 (E8M0 byte 127 everywhere); the
  // per-token scale is applied in the epilogue.
  if (!C::kTiledSfb)
    for (int i = threadIdx.x; i < 128; i += blockDim.x)
      reinterpret_cast<uint32_t*>(smem + C::kOffSFB)[i] = 0x7F7F7F7Fu;
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Constant activation scales into TMEM once, finished before any issuer
  // (each a different thread) runs an MMA that reads them.
  if (!C::kTiledSfb && warp == C::kIssuer0 && lane == 0) {
    const uint64_t sfb_desc = smem_desc(smem_u32(smem + C::kOffSFB), 0, 128, 0);
    tc_cp_32x128b_x4(tmem + C::kColSFB, sfb_desc);
    tc_cp_32x128b_x4(tmem + C::kColSFB + 4, sfb_desc);
    tc_commit(drain + NI);
    int32_t none = 0;
    mbar_wait(drain + NI, 0, timeout_ns, status, kDevTimeout, &none);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Everything above overlaps the previous kernel's tail; the tile list and
  // the activations are that kernel's (or an earlier one's) output.
  // The weight and scale copies need only the tile list.  When it was
  // complete before the previous kernel passed its own wait (early_list:
  // GEMM2, whose list the expansion wrote before GEMM1 started its work, and
  // GEMM1 after the large-batch expansion, whose list the scan wrote before
  // the scatter kernel started) -- each kernel signals its dependents only
  // after its own wait, so this grid starts after that point -- the weight
  // and scale lanes of the producer warps issue their stage's first fill,
  // reading the list through L2, before the producer warps wait with the
  // rest of the CTA: the ring fills while the previous kernels finish.
  constexpr int LPS = C::kLanesPerStage;
  const bool preissue = early_list != 0 && !kChecks && LPS == 3;
  const bool early = preissue && warp < C::kProdWarps;
  if (!early) {
    griddep_wait();
    griddep_launch_dependents();
  }
  const WorkLimits lim = work_limits(status);
  // (producer warps of GEMM2 read the list before their wait: through L2)
  auto tile_at = [&](int i, bool before_wait) -> int4 {
    return before_wait ? __ldcg(tiles + i) : checked_tile(tiles, i, BN, status, lim);
  };
  // The CTA's first tile entry is read together with the tile count (both
  // come from the expansion kernel, and the entry lies inside the list's
  // allocation), so the first copies wait for one round trip, not two.
  const int first_tile = static_cast<int>(blockIdx.x) / MT;
  const int4 first_td = kChecks || first_tile >= max_tiles ? make_int4(0, 0, 0, 0)
                        : early                            ? __ldcg(tiles + first_tile)
                                                           : tiles[first_tile];
  // < 2^31: tiles <= R/16 + E + 1
  const int num_items =
      (early ? __ldcg(num_tiles_p) : checked_num_tiles(num_tiles_p, status, lim)) * MT;

  // ------------------------------------------------------------ producer
  // Stage s belongs to producer warp s % kProdWarps; its LPS = 3 lanes (from
  // lane LPS * (s / kProdWarps)) copy the weight box, the activation box and
  // the scale block (with LPS = 2 the activation lane also copies the scale
  // block).  Each lane arrives on the stage's full barrier with its own byte
  // count, for this CTA's fills f = s, s + STAGES, ... (fill f = K stage
  // f % KS of the CTA's (f / KS)-th item).  Spreading the copies over
  // threads and warps keeps their issue off any single thread's critical
  // path.
  // first_only: issue the stage's first fill only (before the wait) and
  // return whether it did; skip_first: that fill was issued already.
  auto produce = [&](const int s, const int role, const bool first_only,
                     const bool skip_first) -> bool {
    {
      uint32_t phase = 0;
      bool issued = false;
      // fill f = s + j * STAGES: K stage ks of the CTA's it-th item (KS >= STAGES
      // is not assumed; the counters advance without divisions)
      int ks = s % KS, item = blockIdx.x + (s / KS) * gridDim.x;
      // the lane's current item: its tile and first weight box, re-read only
      // when the item changes (runtime divisions stay off the per-fill path)
      int cur_item = -1;
      int4 td = make_int4(0, 0, 0, 0);
      int64_t blk0 = 0;
      while (item < num_items) {
        if (item != cur_item) {
          cur_item = item;
          td = !kChecks && item / MT == first_tile ? first_td : tile_at(item / MT, first_only);
          // prepared weights: one contiguous 128 x 128 box per (expert,
          // M-tile, K stage); box row = ((e * MT + mt) * KS + ks) * 128
          blk0 = (static_cast<int64_t>(td.x) * MT + item % MT) * KS;
        }
        const int64_t blk = blk0 + ks;
        const bool skip = skip_first && !issued;
        if (!skip && !mbar_wait(empty + s, phase ^ 1u, timeout_ns, status, kDevTimeout, abort_flag))
          break;
        if (skip) {
          // issued before the wait
        } else if (role == 0) {
          mbar_arrive_expect_tx(full + s, a_tx_bytes);
          tma_load_2d(smem + C::kOffA + s * C::kABytes, &tmap_w, 0,
                      static_cast<int32_t>(blk * kTileM), full + s);
        } else if (role == 1) {
          // smallest activation box that covers the tile's MMA-N rows
          const int nmma = (td.z + 15) & ~15;
          const int xm = x_map_for(nmma);
          const uint32_t bx = static_cast<uint32_t>(kXBoxRowsAt(xm)) * 128u;
          if constexpr (C::kSplit) {
            // both terms' boxes (hi at K column 128 ks, lo at K + 128 ks of
            // the 2K-wide code rows) and the stage's scale block (the hi
            // term's 512 bytes, then the lo term's)
            mbar_arrive_expect_tx(full + s, (LPS == 2 ? 2 * bx + 512u : 2 * bx) + 1024u);
            uint8_t* b = smem + C::kOffB + s * C::kBBytes;
            tma_load_2d(b, &tmap_x.m[xm], ks * kTileK, td.y, full + s);
            tma_load_2d(b + C::kTermBytes, &tmap_x.m[xm], (KS + ks) * kTileK, td.y, full + s);
            bulk_load(smem + C::kOffSFBs + s * C::kSFBSlot,
                      sfb_tiled + (static_cast<int64_t>(item / MT) * KS + ks) * kSfbTileBytes,
                      1024u, full + s);
          } else {
            // MXFP8: the tile's activation scales for this K stage (one
            // 512-byte block per 128 rows of the MMA-N)
            const uint32_t sfb_bytes = C::kTiledSfb ? (nmma > 128 ? 1024u : 512u) : 0u;
            mbar_arrive_expect_tx(full + s, (LPS == 2 ? bx + 512u : bx) + sfb_bytes);
            tma_load_2d(smem + C::kOffB + s * C::kBBytes, &tmap_x.m[xm], ks * kTileK, td.y,
                        full + s);
            if (C::kTiledSfb)
              bulk_load(smem + C::kOffSFBs + s * C::kSFBSlot,
                        sfb_tiled + (static_cast<int64_t>(item / MT) * KS + ks) * kSfbTileBytes,
                        sfb_bytes, full + s);
          }
          if (LPS == 2)
            tma_load_2d(smem + C::kOffSF + s * C::kSFBytes, &tmap_sf, 0,
                        static_cast<int32_t>(blk), full + s);
        } else {
          mbar_arrive_expect_tx(full + s, 512u);
          tma_load_2d(smem + C::kOffSF + s * C::kSFBytes, &tmap_sf, 0, static_cast<int32_t>(blk),
                      full + s);
        }
        if (first_only) return true;
        issued = true;
        phase ^= 1u;
        ks += STAGES;
        while (ks >= KS) {
          ks -= KS;
          item += gridDim.x;
        }
      }
      if (first_only) return false;
      // Every issued copy must land before the CTA may exit: wait for this
      // stage's last fill (ignores the abort flag, still bounded).
      if (issued) {
        int32_t none = 0;
        mbar_wait(full + s, phase ^ 1u, timeout_ns, status, kDevTimeout, &none);
      }
    }
    return false;
  };

  // Gathering producer warp s (the whole warp, warp-uniform): per fill, wait
  // for the slot; lane 0 copies the weight box and its scales; the 32 lanes
  // copy the tile's nmma rows (row r = token tok[r], K columns 128 ks ..
  // +127) into the slot's 128-byte-swizzled activation box by 16-byte
  // asynchronous copies (row (lane / 8) + 4 i, piece lane % 8), all in
  // flight at once, each lane arriving on the slot's barrier when its copies
  // land (the issuer fences the proxies after its wait).  The token rows are
  // read by each token's k tiles at different times, so they are kept in L2
  // (evict-last) while the weight boxes stream past (evict-first).  first_only /
  // skip_first as in produce (the token list is read only after the grid
  // wait: the previous kernel wrote it).
  auto produce_gather = [&](const int s, const bool first_only, const bool skip_first) -> bool {
    if constexpr (C::kGatherFits && ACT == kActFp8Row && SWIGLU) {
      uint32_t phase = 0;
      bool issued = false;
      int ks = s % KS, item = blockIdx.x + (s / KS) * gridDim.x;
      int cur_item = -1, nmma = 16;
      int4 td = make_int4(0, 0, 0, 0);
      int64_t blk0 = 0;
      int32_t* tok = reinterpret_cast<int32_t*>(smem + C::kOffTok) + s * BN;
      const int c = lane & 7;
      const uint64_t pol_keep = l2_policy_evict_last(), pol_stream = l2_policy_evict_first();
      while (item < num_items) {
        if (item != cur_item) {
          cur_item = item;
          td = !kChecks && item / MT == first_tile ? first_td : tile_at(item / MT, first_only);
          blk0 = (static_cast<int64_t>(td.x) * MT + item % MT) * KS;
          nmma = (td.z + 15) & ~15;
          if (!first_only) {
            // rows past the tile's count repeat its last row (their MMA
            // columns are not stored)
            const int last = max(td.z, 1) - 1;
            __syncwarp();
            for (int r = lane; r < nmma; r += 32)
              tok[r] = __ldg(gather_slot + td.y + min(r, last)) / gather_k;
            __syncwarp();
          }
        }
        const int64_t blk = blk0 + ks;
        const bool skip = skip_first && !issued;
        if (!skip &&
            !mbar_wait_warp(empty + s, phase ^ 1u, timeout_ns, status, kDevTimeout, abort_flag))
          break;
        if (!skip && lane == 0) {
          mbar_arrive_expect_tx(full + s, a_tx_bytes + 512u);
          tma_load_2d_hint(smem + C::kOffA + s * C::kABytes, &tmap_w, 0,
                           static_cast<int32_t>(blk * kTileM), full + s, pol_stream);
          tma_load_2d(smem + C::kOffSF + s * C::kSFBytes, &tmap_sf, 0, static_cast<int32_t>(blk),
                      full + s);
        }
        if (first_only) return true;
        uint8_t* b = smem + C::kOffB + s * C::kBBytes;
        const uint8_t* src = xg + static_cast<int64_t>(ks) * kTileK + 16 * c;
        for (int row = lane >> 3; row < nmma; row += 4)
          cp_async_16_hint(b + row * 128 + ((c ^ (row & 7)) << 4),
                           src + static_cast<int64_t>(tok[row]) * K, pol_keep);
        cp_async_arrive(full + s);   // each lane, once its copies have landed
        issued = true;
        phase ^= 1u;
        ks += STAGES;
        while (ks >= KS) {
          ks -= KS;
          item += gridDim.x;
        }
      }
      if (first_only) return false;
      // every issued copy lands before the CTA may exit (bounded)
      if (issued) {
        int32_t none = 0;
        mbar_wait(full + s, phase ^ 1u, timeout_ns, status, kDevTimeout, &none);
      }
    }
    return false;
  };

  if (warp < C::kProdWarps) {
    const int s = warp + C::kProdWarps * (lane / LPS), role = lane % LPS;
    bool pre = false;
    if (early) {
      if (gather)
        pre = produce_gather(warp, true, false);
      else if (s < STAGES && role != 1)
        pre = produce(s, role, true, false);
      __syncwarp();
      griddep_wait();
      griddep_launch_dependents();
    }
    if (gather)
      produce_gather(warp, false, pre);
    else if (s < STAGES)
      produce(s, role, false, pre);
  } else if (warp < C::kIssuer0 + NI) {
    // ------------------------------------------------------------ MMA issuers
    // Each tcgen05 instruction occupies its issuing warp (measured ~310
    // cycles per stage of one copy + 4 MMAs from a warp-uniform loop, ~510
    // from a loop that only lane 0 runs, independent of N up to 128), so with
    // small token tiles one issuing warp cannot keep pace with the weight
    // stream.
    // Issuer i (warp kIssuer0 + i) takes fills f = i, i + ni, i + 2 ni, ... -- i.e.
    // the stages s with s % ni == i -- and accumulates its K stages of an item
    // into its own TMEM accumulator; the epilogue sums the ni partials.
    // Every descriptor is precomputed: stage s and K sub-step kk only add
    // constant start-address offsets (address >> 4 lives in the low 14 bits).
    // The whole warp runs the loop (uniform control flow); one elected lane
    // issues each tcgen05 instruction.
    const int i = warp - C::kIssuer0;
    if (i < ni) {
      const uint64_t adesc0 = smem_desc(smem_u32(smem + C::kOffA), 0, 1024, 2);
      const uint64_t bdesc0 = smem_desc(smem_u32(smem + C::kOffB), 0, 1024, 2);
      const uint64_t sdesc0 = smem_desc(smem_u32(smem + C::kOffSF), 0, 128, 0);
      const uint64_t sbdesc0 = smem_desc(smem_u32(smem + C::kOffSFBs), 0, 128, 0);
      // One stage, from one elected lane in one block: weight scales (and
      // per-stage activation scales) into TMEM, the 4 MMAs of its 128 K (the
      // first of an item's first stage overwrites the accumulator; split:
      // then the lo term's 4 MMAs into the same accumulator), and the commit
      // that frees the slot when they complete.  Electing once per stage
      // instead of once per instruction took DSV3 T=4096 from 1557 to 1532
      // us.
      auto issue_stage = [&](int stage, uint32_t d_tmem, uint32_t id0, int nmma, bool first) {
        const uint32_t sfa = tmem + static_cast<uint32_t>(C::kColSFA + 4 * stage);
        const uint64_t sfa_src = sdesc0 + static_cast<uint64_t>(stage * (C::kSFBytes >> 4));
        const uint64_t ad = adesc0 + static_cast<uint64_t>(stage * (C::kABytes >> 4));
        const uint64_t bd = bdesc0 + static_cast<uint64_t>(stage * (C::kBBytes >> 4));
        const uint32_t acc0 = first ? 0u : 1u, bar = smem_u32(empty + stage);
        if constexpr (!C::kTiledSfb) {
          tc_stage_mx4_warp(d_tmem, ad, bd, id0, sfa, sfa_src, tmem + C::kColSFB, acc0, bar);
        } else {
          const uint32_t sfb = tmem + static_cast<uint32_t>(C::kColSFB + 8 * stage);
          const uint64_t sfb_src = sbdesc0 + static_cast<uint64_t>(stage * (C::kSFBSlot >> 4));
          if constexpr (C::kSplit)
            tc_stage_split_warp(d_tmem, ad, bd, bd + static_cast<uint64_t>(C::kTermBytes >> 4),
                                id0, sfa, sfa_src, sfb, sfb_src, acc0, bar);
          else
            tc_stage_mx4_sfb_warp(d_tmem, ad, bd, id0, sfa, sfa_src, sfb, sfb_src,
                                  nmma > 128 ? 1u : 0u, acc0, bar);
        }
      };
      if constexpr (NI == 1) {
        // One issuer (prefill tiles): items in order, an item's K stages in
        // order.  The issuing warp's serial instruction stream bounds the
        // MMA rate on these tiles, so the loop carries nothing but the stage
        // and phase counters.
        uint32_t stage = 0, phase = 0;
        int fidx = 0;
        bool ok = true;
        for (int item = blockIdx.x, it = 0; ok && item < num_items;
             item += static_cast<int>(gridDim.x), ++it) {
          const int4 td = checked_tile(tiles, item / MT, BN, status, lim);
          const int nmma = (td.z + 15) & ~15;
          const uint32_t id0 = idesc_mx(kAFmt, 0, static_cast<uint32_t>(nmma), 0, 0);
          const int acc = it % NB;
          if (!mbar_wait_warp(tempty + acc, static_cast<uint32_t>((it / NB) & 1) ^ 1u, timeout_ns,
                              status, kDevTimeout, abort_flag))
            break;
          tc_fence_after();
          const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
          for (int ks = 0; ks < KS; ++ks) {
            if (!mbar_wait_warp(full + stage, phase, timeout_ns, status, kDevTimeout, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (gather) fence_proxy_async_smem();   // gathered rows: generic-proxy copies
            issue_stage(static_cast<int>(stage), d_tmem, id0, nmma, ks == 0);
            if (prefetch_stages > 0 && lane == 0) *progress = fidx;
            ++fidx;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) tc_commit_warp(tfull + acc);   // the item's accumulator is final
        }
      } else {
        int stage = i % STAGES, ks = i % KS, it = i / KS;   // ni <= KS, so it == 0
        int nmma = 16, fidx = i;
        uint32_t phase = (i / STAGES) & 1;
        bool new_item = true;
        uint32_t d_tmem = 0, id0 = 0;
        int acc = 0;
        while (blockIdx.x + it * static_cast<int>(gridDim.x) < num_items) {
          if (new_item) {
            const int item = blockIdx.x + it * gridDim.x;
            const int4 td = checked_tile(tiles, item / MT, BN, status, lim);
            nmma = (td.z + 15) & ~15;
            id0 = idesc_mx(kAFmt, 0, static_cast<uint32_t>(nmma), 0, 0);
            acc = it % NB;
            if (!mbar_wait_warp(tempty + acc, static_cast<uint32_t>((it / NB) & 1) ^ 1u, timeout_ns,
                                status, kDevTimeout, abort_flag))
              break;
            tc_fence_after();
            d_tmem = tmem + static_cast<uint32_t>((acc * NI + i) * BN);
          }
          if (!mbar_wait_warp(full + stage, phase, timeout_ns, status, kDevTimeout, abort_flag))
            break;
          tc_fence_after();
          if (gather) fence_proxy_async_smem();
          issue_stage(stage, d_tmem, id0, nmma, new_item);
          if (i == 0 && lane == 0) *progress = fidx;
          fidx += ni;
          stage += ni;
          if (stage >= STAGES) {
            stage -= STAGES;
            phase ^= 1u;
          }
          ks += ni;
          new_item = false;
          while (ks >= KS) {
            ks -= KS;
            ++it;
            new_item = true;
          }
          if (new_item) tc_commit_warp(tfull + acc);   // this issuer's share of the item is queued
        }
      }
      // No MMA or TMEM copy may still be running when TMEM is freed.
      tc_commit_warp(drain + i);
      int32_t none = 0;
      mbar_wait_warp(drain + i, 0, timeout_ns, status, kDevTimeout, &none);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    if (warp < C::kIssuer0 + NI + kEpiWarps) {
      const EpiSched sch{static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), MT, 1, 0, 0u};
      epilogue_loop<BN, NI, NB, SWIGLU>(C::kIssuer0 + NI, ni, tiles, num_items, sch, tfull, tempty,
                                         tmem, row_scale, out, out_ld, timeout_ns, status,
                                         abort_flag, SWIGLU ? CombineArgs{} : cmb);
    } else if (prefetch_stages > 0) {
      // ---------------------------------------------------------- prefetcher
      // Optional: asks L2 for the weight box of fill g while the first issuer
      // has consumed fills up to g - prefetch_stages (plain prefetch
      // instructions, 128 bytes per lane-instruction, outside the TMA
      // unit), so that box's TMA load later hits L2.  It paces itself on a
      // progress word the first issuer publishes -- no barrier -- and stops
      // quietly when the pipeline does; a prefetch changes no result.
      int total = 0;
      for (int it2 = blockIdx.x; it2 < num_items; it2 += gridDim.x) total += KS;
      int g = STAGES < total ? STAGES : total, kp = g % KS;
      int itp = blockIdx.x + (g / KS) * static_cast<int>(gridDim.x);
      int last_seen = -2;
      uint64_t t_last = globaltimer_ns();
      while (g < total) {
        const int p = *progress;
        if (g <= p + prefetch_stages) {
          const int64_t bp =
              (static_cast<int64_t>(checked_tile(tiles, itp / MT, BN, status, lim).x) * MT +
               itp % MT) * KS + kp;
          const uint8_t* box = w_base + bp * a_tx_bytes;
          for (uint32_t off = static_cast<uint32_t>(lane) * 128u; off < a_tx_bytes;
               off += 32u * 128u)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(box + off));
          ++g;
          if (++kp == KS) {
            kp = 0;
            itp += gridDim.x;
          }
          continue;
        }
        if (*abort_flag) break;
        const uint64_t now = globaltimer_ns();
        if (p != last_seen) {
          last_seen = p;
          t_last = now;
        } else if (now - t_last > timeout_ns) {
          break;
        }
        __nanosleep(64);   // idle: leave the issue slots to the working warps
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kIssuer0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, int STAGES, int NI, int NB, bool SWIGLU, int ACT>
cudaError_t launch_variant(const GemmArgs& a, cudaStream_t s) {
  using C = GemmCfg<BN, STAGES, NI, NB, ACT>;
  auto kern = grouped_gemm_kernel<BN, STAGES, NI, NB, SWIGLU, ACT>;
  static DeviceOnce smem_set;   // per instantiation and device
  const cudaError_t e = set_smem_limit_once(kern, C::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  XMaps xm;
  for (int i = 0; i < kNumXMaps; ++i) xm.m[i] = a.tmap_x[i];
  if (a.gather_slot && !(C::kGatherFits && ACT == kActFp8Row && SWIGLU)) return cudaErrorInvalidValue;
  return launch_pdl(kern, dim3(a.num_sms), dim3(C::kThreads), C::kSmemBytes, s, *a.tmap_w, xm,
                    *a.tmap_sf, a.tiles, a.num_tiles, a.row_scale,
                    static_cast<__nv_bfloat16*>(a.out), a.m_per_expert, a.k, a.out_ld, a.status,
                    a.timeout_ns, a.a_tx_bytes, a.prefetch_stages, a.sfb_tiled, a.w_base,
                    a.max_tiles, a.early_list ? 1 : 0, a.gather_slot, a.gather_k, a.gather_x,
                    CombineArgs{a.cmb_cnt, a.cmb_slot, a.cmb_row_of, a.cmb_wts,
                                static_cast<__nv_bfloat16*>(a.cmb_out), a.cmb_k,
                                a.m_per_expert / kTileM});
}

}  // namespace

// Variants: <token tile BN, pipeline stages, MMA issuers NI, accumulator
// buffers NB>, then the stages and issuers of the MXFP8 instantiation (its
// stages also hold the activation scales, so the deepest rings lose a
// stage).
//   1: decode tiles of <= 32 tokens, 10 stages, 5 issuers;
//   2: prefill tiles of <= 224 tokens, 5 stages;
//   3: decode tiles of <= 16 tokens, 12 stages (the smallest stage, so the
//      most weight bytes in flight), 6 issuers;
//   4: tiles of <= 224 tokens with 2 issuers and one accumulator buffer (the
//      epilogue no longer overlaps the next item's MMAs);
//   5: tiles of <= 160 tokens, 6 stages;
//   6: tiles of <= 160 tokens on CTA pairs (gemm_pair.cu), 8 stages.
#define MOE_GEMM_VARIANTS(X)          \
  X(1, kDecodeBN, 10, 5, 2, 10, 5)    \
  X(2, kPrefillBN, 5, 1, 2, 4, 1)     \
  X(3, kTinyBN, 12, 6, 2, 10, 5)      \
  X(4, kPrefillBN, 4, 2, 1, 4, 2)     \
  X(5, kMidBN, 6, 1, 2, 6, 1)

// The split activations (W4A16) carry two terms per stage, so their tiles
// stop at kW4A16BN tokens: variants 1 and 3 keep their tile size with
// <BN, stages, issuers, buffers> below; 2, 4, 5 and 6 run the 64-token tile.
#define MOE_SPLIT_VARIANTS(X)  \
  X(3, kTinyBN, 10, 5, 2)      \
  X(1, kDecodeBN, 8, 4, 2)     \
  X(5, kW4A16BN, 6, 3, 2)

namespace {
int split_variant(int variant) { return variant == 1 || variant == 3 ? variant : 5; }
}  // namespace

int gemm_tile_tokens(int variant, int act) {
  if (act == kActSplit) {
    switch (split_variant(variant)) {
#define MOE_S(v, bn, st, ni, nb) \
  case v:                        \
    return bn;
      MOE_SPLIT_VARIANTS(MOE_S)
#undef MOE_S
      default:
        return kW4A16BN;
    }
  }
  if (variant == 6) return kPairBN;
  switch (variant) {
#define MOE_X(v, bn, st, ni, nb, st8, ni8) \
  case v:                                  \
    return bn;
    MOE_GEMM_VARIANTS(MOE_X)
#undef MOE_X
    default:
      return kMidBN;
  }
}

bool gemm_gather_supported(int variant) {
  switch (variant) {
#define MOE_X(v, bn, st, ni, nb, st8, ni8) \
  case v:                                  \
    return GemmCfg<bn, st, ni, nb, kActFp8Row>::kGatherFits;
    MOE_GEMM_VARIANTS(MOE_X)
#undef MOE_X
    default:
      return false;
  }
}

cudaError_t launch_gemm(bool swiglu, int variant, const GemmArgs& a, cudaStream_t s) {
  if (a.act == kActSplit) {
    switch (split_variant(variant)) {
#define MOE_S(v, bn, st, ni, nb)                                              \
  case v:                                                                     \
    return swiglu ? launch_variant<bn, st, ni, nb, true, kActSplit>(a, s)     \
                  : launch_variant<bn, st, ni, nb, false, kActSplit>(a, s);
      MOE_SPLIT_VARIANTS(MOE_S)
#undef MOE_S
      default:
        return cudaErrorInvalidValue;
    }
  }
  // Variant 6: CTA pairs where the operands allow (W4A8, an even number of
  // M-tiles), else the one-CTA kernel with the same 160-token tiles.
  static_assert(kPairBN == kMidBN, "variant 6 falls back to variant 5's tile size");
  if (variant == 6) {
    if (gemm_pair_supported(a.m_per_expert, a.act) && a.tmap_x_pair && a.num_sms >= 2)
      return launch_gemm_pair(swiglu, a, s);
    variant = 5;
  }
  switch (variant) {
#define MOE_X(v, bn, st, ni, nb, st8, ni8)                                        \
  case v:                                                                         \
    if (a.act == kActMxfp8)                                                       \
      return swiglu ? launch_variant<bn, st8, ni8, nb, true, kActMxfp8>(a, s)     \
                    : launch_variant<bn, st8, ni8, nb, false, kActMxfp8>(a, s);   \
    return swiglu ? launch_variant<bn, st, ni, nb, true, kActFp8Row>(a, s)        \
                  : launch_variant<bn, st, ni, nb, false, kActFp8Row>(a, s);
    MOE_GEMM_VARIANTS(MOE_X)
#undef MOE_X
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
