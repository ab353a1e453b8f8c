// gemm_bf16.cu -- the grouped GEMM of the W4A16 mode: MXFP4 weights x bf16
// activations on the sm_103a tensor cores (tcgen05 .kind::f16, TMEM
// accumulators).
//
// Pages cited (title and section):
//   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
//           MXFP4xFP8 CUTLASS MoE backend for SM90": title and Description
//           (the MXFP4 x BF16 MoE GEMM: bf16 activations fed unquantised,
//           MXFP4 weights dequantised inside the kernel).
//
// The tensor cores have no mixed FP4 x BF16 MMA, so the weights are
// converted on the fly, in sub-stages of 64 K: the packed E2M1 codes of 128
// weight rows x 64 K (half of a prepared 128 x 128 box, 32 bytes per row)
// and the box's E8M0 scales land in a raw shared-memory slot; transform
// warps turn them into bf16 values e2m1 * 2^(scale - 127) -- exact in bf16
// (a power of two times at most two significant bits) -- and store them
// straight into TMEM, where the MMA (.kind::f16) reads its A operand; only
// the bf16 activation atom (B) is read from shared memory.  Keeping the
// converted weights in TMEM frees shared memory for a deep raw ring and
// gives the conversion 8 slots to run ahead in.  Everything else (tile
// list, swap-AB orientation, persistent static striding, epilogue) is the
// FP8 GEMM's.
//
// Roles: warps 0..2 = TMA producers (slot s in warp s % 3: one lane for the
// weight half-box + scales into raw slot s, one for the activation atom
// into activation slot s); the next NI warps = MMA issuers (warp-uniform, one elected lane issues; issuer i takes
// the sub-stages g = i mod NI into its own accumulator); the next 16 warps
// = transform, four groups of four (group p converts the sub-stages
// g = p mod 4, warp w of the group the rows of TMEM lane quarter w % 4); the
// last 4 warps = epilogue, one per lane quarter.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

// Transform warps: four groups of four (group g % 4 converts sub-stage g,
// warp w of the group the rows of TMEM lane quarter w % 4), so each group
// has four sub-stages of time per conversion.
constexpr int kXfGroups = 4;
constexpr int kTransformWarps = 4 * kXfGroups;
// The W4A16 tiles hold at most 64 tokens: one epilogue warp per quarter.
constexpr int kBf16EpiWarps = 4;
// Producer warps: slot s is served by warp s % 3 (lanes of one warp waiting
// on different slots' barriers serialise), two lanes per slot.
constexpr int kBf16ProdWarps = 3;
constexpr int kBf16Issuers = 2;

template <int BN, int S, int QA>
struct Bf16Cfg {
  static_assert(BN % 16 == 0 && BN <= 128, "token tile of the W4A16 GEMM: 16..128 rows");
  static_assert(2 * ((S + kBf16ProdWarps - 1) / kBf16ProdWarps) <= 32,
                "producer lanes must fit the producer warps");
  // slot s (raw, activation) and TMEM slot a always belong to one issuer and
  // one transform pair, so each barrier is waited on in phase order by the
  // same threads
  static_assert(S % kBf16Issuers == 0 && QA % kBf16Issuers == 0 && S % kXfGroups == 0 &&
                    QA % kXfGroups == 0,
                "slots must map to single issuers and transform groups");
  static constexpr int kRawBytes = kTileM * 32;      // packed E2M1, 64 K per row
  static constexpr int kSFBytes = 512;               // 128 rows x 4 E8M0 bytes (128 K)
  static constexpr int kBBytes = BN * 128;           // 64 bf16 of K per token row
  static constexpr int kOffRaw = 0;
  static constexpr int kOffB = kOffRaw + S * kRawBytes;
  static constexpr int kOffSF = kOffB + S * kBBytes;
  // code byte -> bf16x2 table, one copy per shared-memory bank: entry b of
  // lane l at word 32 b + l, so a warp's lookups never conflict
  static constexpr int kOffLut = kOffSF + S * kSFBytes;
  static constexpr int kNumBars = 4 * S + 2 * QA + 2 * 2 + kBf16Issuers;
  static constexpr int kOffBar = kOffLut + 256 * 32 * 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + base alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
  static constexpr int kFirstIssuer = kBf16ProdWarps;   // owns TMEM
  static constexpr int kFirstXfWarp = kFirstIssuer + kBf16Issuers;
  static constexpr int kFirstEpiWarp = kFirstXfWarp + kTransformWarps;
  static constexpr int kThreads = 32 * (kFirstEpiWarp + kBf16EpiWarps);
  // TMEM: 2 accumulator buffers x NI partials x BN columns, then QA slots of
  // converted weights, 32 columns each (128 rows x 64 bf16)
  static constexpr int kColA = 2 * kBf16Issuers * BN;
  static constexpr int kColsUsed = kColA + 32 * QA;
  static_assert(kColsUsed <= 512, "TMEM budget exceeded");
  static constexpr int kTmemCols = kColsUsed <= 256 ? 256 : 512;
};

// Instruction descriptor of .kind::f16 with bf16 A and B, fp32 accumulate,
// M = 128, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// D (+)= A x B^T with A read from TMEM (128 lanes = rows; K = 16 bf16 in 8
// columns, two per column, the lower K index in the low half) and B from
// shared memory; one elected lane of the warp issues.
__device__ __forceinline__ void tc_mma_f16_ts_warp(uint32_t d_tmem, uint32_t a_tmem,
                                                   uint64_t bdesc, uint32_t idesc,
                                                   uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Each thread of the warp writes 32 consecutive 32-bit TMEM columns of its
// lane (the warp's lane quarter), then waits until the stores are done.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Value of each E2M1 code (sign, 2-bit exponent with bias 1, 1-bit
// mantissa; OCP MX v1.0), as a float.
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t mag = code & 7u;
  // magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 = (2 + m) * 2^(e - 2) for e > 0,
  // m * 0.5 for e = 0
  const uint32_t e = mag >> 1, m = mag & 1u;
  const float v = e == 0 ? 0.5f * static_cast<float>(m)
                         : static_cast<float>(2u + m) * __uint_as_float((125u + e) << 23);
  return (code & 8u) ? -v : v;
}

// bf16 of the E8M0 scale 2^(sb - 127), twice: the exponent field is sb
// (sb = 0: the subnormal 2^-127; sb = 255: NaN).
__device__ __forceinline__ __nv_bfloat162 e8m0_bf16x2(uint32_t sb) {
  const uint16_t bits =
      sb == 0 ? 0x0040u : sb == 255 ? 0x7FC0u : static_cast<uint16_t>(sb << 7);
  __nv_bfloat162 r;
  r.x = __ushort_as_bfloat16(bits);
  r.y = r.x;
  return r;
}

template <int BN, int S, int QA, bool SWIGLU>
__global__ void __launch_bounds__(Bf16Cfg<BN, S, QA>::kThreads, 1)
    grouped_gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmap_w,
                             const __grid_constant__ XMaps tmap_x,
                             const __grid_constant__ CUtensorMap tmap_sf,
                             const int4* __restrict__ tiles,
                             const int32_t* __restrict__ num_tiles_p,
                             __nv_bfloat16* __restrict__ out, int m_per_expert, int K,
                             int out_ld, int32_t* __restrict__ status, uint64_t timeout_ns) {
  using C = Bf16Cfg<BN, S, QA>;
  constexpr int NI = kBf16Issuers;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* raw_empty = raw_full + S;
  uint64_t* b_full = raw_empty + S;
  uint64_t* b_empty = b_full + S;
  uint64_t* a_full = b_empty + S;
  uint64_t* a_empty = a_full + QA;
  uint64_t* tfull = a_empty + QA;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MT = m_per_expert / kTileM, KS = K / kTileK;
  const int KH = 2 * KS;   // 64-K sub-stages per item (>= 2 = NI)

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(raw_full + s, 1);
      mbar_init(raw_empty + s, 4);   // the four quarter warps of its transform group
      mbar_init(b_full + s, 1);
      mbar_init(b_empty + s, 1);
    }
    for (int a = 0; a < QA; ++a) {
      mbar_init(a_full + a, 4);      // each quarter of the 128 rows stored
      mbar_init(a_empty + a, 1);     // the MMAs that read it completed
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, NI);                     // every issuer commits its share
      mbar_init(tempty + a, kBf16EpiWarps);
    }
    for (int i = 0; i < NI; ++i) mbar_init(drain + i, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_sf);
    for (int i = 0; i < kNumXMaps; ++i) prefetch_tmap(&tmap_x.m[i]);
  }
  if (warp == C::kFirstIssuer) tmem_alloc(tmem_slot, C::kTmemCols);
  // Code byte -> the bf16 pair (low nibble = even k) of its two E2M1 values,
  // replicated per bank.
  for (int w = threadIdx.x; w < 256 * 32; w += blockDim.x) {
    const int b = w >> 5;
    const __nv_bfloat162 pr = __floats2bfloat162_rn(e2m1_value(b & 0xF), e2m1_value(b >> 4));
    reinterpret_cast<__nv_bfloat162*>(smem + C::kOffLut)[w] = pr;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();
  griddep_launch_dependents();
  const WorkLimits lim = work_limits(status);
  const int num_items = checked_num_tiles(num_tiles_p, status, lim) * MT;

  if (warp < kBf16ProdWarps) {
    // ------------------------------------------------------------ producer
    // Slot s belongs to warp s % 3: its lane 2 (s / 3) fills raw slot s for
    // this CTA's sub-stages g = s, s + S, ... (sub-stage g = 64-K half
    // (g % KH) % 2 of the 128-K box (g % KH) / 2 of the CTA's (g / KH)-th
    // item) and the next lane fills activation slot s.
    const int s = warp + kBf16ProdWarps * (lane >> 1);
    if (s < S) {
      const bool is_w = (lane & 1) == 0;
      uint32_t phase = 0;
      bool issued = false;
      int kh = s % KH, item = blockIdx.x + (s / KH) * gridDim.x;
      uint64_t* full = is_w ? raw_full + s : b_full + s;
      uint64_t* empty = is_w ? raw_empty + s : b_empty + s;
      while (item < num_items) {
        const int mt = item % MT;
        const int4 td = checked_tile(tiles, item / MT, BN, status, lim);
        if (!mbar_wait(empty, phase ^ 1u, timeout_ns, status, kDevTimeout, abort_flag)) break;
        if (is_w) {
          const int64_t blk = (static_cast<int64_t>(td.x) * MT + mt) * KS + (kh >> 1);
          mbar_arrive_expect_tx(full, static_cast<uint32_t>(C::kRawBytes) + 512u);
          tma_load_2d(smem + C::kOffRaw + s * C::kRawBytes, &tmap_w, (kh & 1) * 32,
                      static_cast<int32_t>(blk * kTileM), full);
          tma_load_2d(smem + C::kOffSF + s * C::kSFBytes, &tmap_sf, 0, static_cast<int32_t>(blk),
                      full);
        } else {
          // the smallest box covering the MMA-N rows, 64 K elements
          const int nmma = (td.z + 15) & ~15;
          const int xm = x_map_for(nmma);
          mbar_arrive_expect_tx(full, static_cast<uint32_t>(kXBoxRowsAt(xm)) * 128u);
          tma_load_2d(smem + C::kOffB + s * C::kBBytes, &tmap_x.m[xm], kh * 64, td.y, full);
        }
        issued = true;
        phase ^= 1u;
        kh += S;
        while (kh >= KH) {
          kh -= KH;
          item += gridDim.x;
        }
      }
      if (issued) {
        int32_t none = 0;
        mbar_wait(full, phase ^ 1u, timeout_ns, status, kDevTimeout, &none);
      }
    }
  } else if (warp < C::kFirstXfWarp) {
    // ------------------------------------------------------------ MMA issuers
    const int i = warp - C::kFirstIssuer;
    const uint64_t bdesc0 = smem_desc(smem_u32(smem + C::kOffB), 0, 1024, 2);
    int g = i, kh = i, it = 0;
    bool new_item = true;
    uint32_t d_tmem = 0, id = 0;
    int acc = 0;
    while (blockIdx.x + it * static_cast<int>(gridDim.x) < num_items) {
      if (new_item) {
        const int item = blockIdx.x + it * gridDim.x;
        id = idesc_bf16(
            static_cast<uint32_t>((checked_tile(tiles, item / MT, BN, status, lim).z + 15) & ~15));
        acc = it & 1;
        if (!mbar_wait_warp(tempty + acc, static_cast<uint32_t>((it >> 1) & 1) ^ 1u, timeout_ns,
                            status, kDevTimeout, abort_flag))
          break;
        tc_fence_after();
        d_tmem = tmem + static_cast<uint32_t>((acc * NI + i) * BN);
      }
      const int s = g % S, a = g % QA;
      if (!mbar_wait_warp(a_full + a, static_cast<uint32_t>((g / QA) & 1), timeout_ns, status,
                          kDevTimeout, abort_flag))
        break;
      if (!mbar_wait_warp(b_full + s, static_cast<uint32_t>((g / S) & 1), timeout_ns, status,
                          kDevTimeout, abort_flag))
        break;
      tc_fence_after();
      const uint32_t at = tmem + static_cast<uint32_t>(C::kColA + 32 * a);
      const uint64_t bd = bdesc0 + static_cast<uint64_t>((s * C::kBBytes) >> 4);
#pragma unroll
      for (uint32_t kk = 0; kk < 4; ++kk)   // K = 16 bf16 per MMA: 8 TMEM columns, 32 smem bytes
        tc_mma_f16_ts_warp(d_tmem, at + 8 * kk, bd + 2 * kk, id, (!new_item || kk > 0) ? 1u : 0u);
      tc_commit_warp(a_empty + a);
      tc_commit_warp(b_empty + s);
      g += NI;
      kh += NI;
      new_item = false;
      if (kh >= KH) {   // NI <= KH: at most one item boundary per step
        kh -= KH;
        ++it;
        new_item = true;
        tc_commit_warp(tfull + acc);
      }
    }
    tc_commit_warp(drain + i);
    int32_t none = 0;
    mbar_wait_warp(drain + i, 0, timeout_ns, status, kDevTimeout, &none);
  } else if (warp < C::kFirstEpiWarp) {
    // ------------------------------------------------------------ transform
    // Transform warp w (quarter q = warp % 4, group p) converts, for the
    // sub-stages g = p, p + 4, ..., the 32 rows r = 32 q + lane: lane l reads
    // its row's 32 code bytes and two scale bytes, turns each code byte into
    // a bf16 pair through the shared table (this lane's bank copy: no
    // conflicts), applies the 32-K block's scale with one exact bf16x2
    // multiply, and stores the row's 64 values into 32 columns of its TMEM
    // lane in TMEM slot g % QA.
    const int q = warp & 3, p = (warp - C::kFirstXfWarp) >> 2;   // quarter, group
    const int r = 32 * q + lane;
    const __nv_bfloat162* lutl = reinterpret_cast<const __nv_bfloat162*>(smem + C::kOffLut) + lane;
    const uint32_t tlane = static_cast<uint32_t>(32 * q) << 16;
    int total = 0;
    for (int item = blockIdx.x; item < num_items; item += gridDim.x) total += KH;
    for (int g = p; g < total; g += kXfGroups) {
      const int s = g % S, a = g % QA;
      if (!mbar_wait_warp(raw_full + s, static_cast<uint32_t>((g / S) & 1), timeout_ns, status,
                          kDevTimeout, abort_flag))
        break;
      if (!mbar_wait_warp(a_empty + a, static_cast<uint32_t>((g / QA) & 1) ^ 1u, timeout_ns,
                          status, kDevTimeout, abort_flag))
        break;
      tc_fence_after();
      const uint8_t* raw = smem + C::kOffRaw + s * C::kRawBytes + 32 * r;
      const uint8_t* sf = smem + C::kOffSF + s * C::kSFBytes;
      const int half = g & 1;   // the 64-K half of the 128-K box ((g % KH) & 1: KH is even)
      const uint4 c0 = *reinterpret_cast<const uint4*>(raw);
      const uint4 c1 = *reinterpret_cast<const uint4*>(raw + 16);
      const int sfo = 16 * (r & 31) + 4 * (r >> 5) + 2 * half;
      const __nv_bfloat162 s0 = e8m0_bf16x2(sf[sfo]), s1 = e8m0_bf16x2(sf[sfo + 1]);
      // the raw slot has been read: its producer may refill it
      __syncwarp();
      if (lane == 0) mbar_arrive(raw_empty + s);
      const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      uint32_t v[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {   // code byte c = K elements 2c, 2c + 1
        // byte c & 3 of the word moved to the low byte (one byte permute);
        // this lane's table copy is lutl[32 * byte]
        const uint32_t byte = __byte_perm(cw[c >> 2], 0u, 0x4440u + static_cast<uint32_t>(c & 3));
        const __nv_bfloat162 pr = __hmul2(lutl[byte << 5], c < 16 ? s0 : s1);
        v[c] = *reinterpret_cast<const uint32_t*>(&pr);
      }
      tmem_st_32x32b_x32(tmem + tlane + static_cast<uint32_t>(C::kColA + 32 * a), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(a_full + a);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const EpiSched sch{static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), MT, 1, 0, 0u};
    epilogue_loop<BN, NI, 2, SWIGLU, kBf16EpiWarps>(C::kFirstEpiWarp, NI, tiles, num_items, sch,
                                                    tfull, tempty, tmem, nullptr, out, out_ld,
                                                    timeout_ns, status, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kFirstIssuer) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, int S, int QA, bool SWIGLU>
cudaError_t launch_bf16_variant(const GemmArgs& a, cudaStream_t s) {
  using C = Bf16Cfg<BN, S, QA>;
  auto kern = grouped_gemm_bf16_kernel<BN, S, QA, SWIGLU>;
  static DeviceOnce smem_set;   // per instantiation and device
  const cudaError_t e = set_smem_limit_once(kern, C::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  XMaps xm;
  for (int i = 0; i < kNumXMaps; ++i) xm.m[i] = a.tmap_x[i];
  return launch_pdl(kern, dim3(a.num_sms), dim3(C::kThreads), C::kSmemBytes, s, *a.tmap_w, xm,
                    *a.tmap_sf, a.tiles, a.num_tiles, static_cast<__nv_bfloat16*>(a.out),
                    a.m_per_expert, a.k, a.out_ld, a.status, a.timeout_ns);
}

}  // namespace

// W4A16: 64-token tiles, 12 raw/activation slots, 8 TMEM slots of converted
// weights (64 K each).
cudaError_t launch_gemm_bf16(bool swiglu, const GemmArgs& a, cudaStream_t s) {
  return swiglu ? launch_bf16_variant<kW4A16BN, 12, 8, true>(a, s)
                : launch_bf16_variant<kW4A16BN, 12, 8, false>(a, s);
}

}  // namespace moe
