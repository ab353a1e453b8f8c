// moe_internal.h -- launch helpers shared by the library's translation units
// (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <utility>

#include "../../include/moe.h"

namespace moe {

// Device status codes written to the workspace status word (match moe_status).
constexpr int32_t kDevTimeout = -6;
constexpr int32_t kDevCheckFailed = -7;   // MOE_ERR_DEVICE_CHECK

// Checked builds (-DMOE_CHECKS, libmoe_checked.so) validate the device-built
// work map where the GEMMs consume it; release builds compile the checks
// away.  The first kernel of a forward records the expanded row count R and
// the expert count E in status[2] and status[3] for them.
#ifdef MOE_CHECKS
constexpr bool kChecks = true;
#else
constexpr bool kChecks = false;
#endif

// One-time, per-device setup of a kernel: function attributes such as the
// dynamic shared-memory limit belong to the kernel as loaded on one device,
// so a process that drives several GPUs sets them on each.  A launcher keeps
// one table per kernel instantiation (static storage, zero-initialised);
// the entry for the current device holds 0 until the setup has succeeded.
constexpr int kMaxDevices = 64;
using DeviceOnce = std::atomic<int>[kMaxDevices];

// Current device's entry of `table` (null when the ordinal is out of range).
inline std::atomic<int>* device_entry(DeviceOnce& table, cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  return &table[dev];
}

// Raises the dynamic shared-memory limit of `kern` to `bytes` on the current
// device, once per device.
template <typename... KArgs>
cudaError_t set_smem_limit_once(void (*kern)(KArgs...), int bytes, DeviceOnce& table) {
  cudaError_t e;
  std::atomic<int>* done = device_entry(table, &e);
  if (!done) return e;
  if (done->load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done->store(1, std::memory_order_release);
  return e;
}

// Launches `kern` with programmatic stream serialisation (PDL): the kernel may
// begin while its stream predecessor finishes; every kernel of this library
// calls griddep_wait() before it reads a predecessor's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Largest token count that uses the one-kernel small-batch expansion
// (expand_small_kernel) instead of scan + quant_scatter.  Each of its T
// blocks recounts all T * k routed ids, so its cost grows with T^2: above
// 256 tokens the three-kernel path is cheaper (DSV3 T=512: 26.8 us in the
// one kernel).
constexpr int kSmallT = MOE_SMALL_BATCH_TOKENS;

// Largest token count that routes, expands and quantises in one single-CTA
// kernel (route_expand_tiny_kernel; W4A8 only): one warp per token.
constexpr int kTinyT = MOE_TINY_BATCH_TOKENS;

// Tokens per routing chunk: the unit of the per-chunk expert histogram that
// makes the expert-major scatter deterministic (stable in token order).
constexpr int kRouteChunk = 32;

// GEMM tiling: weights fill MMA-M = 128 (one M-tile), tokens fill MMA-N.
constexpr int kTileM = 128;
constexpr int kTileK = 128;          // K elements per pipeline stage
constexpr int kDecodeBN = 32;        // max tokens per tile, decode variant
constexpr int kTinyBN = 16;          // max tokens per tile, 16-token decode variant
constexpr int kPrefillBN = 224;      // max tokens per tile, prefill variant
constexpr int kMidBN = 160;          // max tokens per tile, 6-stage prefill variant
constexpr int kW4A16BN = 64;         // max tokens per tile of the split (W4A16) GEMM

// Activation box heights (rows) of the GEMM's activation tensor maps:
// 16, 32, 64, 96, ..., 224.
constexpr int kNumXMaps = 8;
__host__ __device__ constexpr int kXBoxRowsAt(int i) { return i == 0 ? 16 : 32 * i; }
// CTA-pair GEMM (gemm_pair.cu): token tiles of up to kPairBN rows, each CTA
// staging half a tile through maps with box heights 16, 32, ..., 128 rows.
constexpr int kPairBN = 160;
constexpr int kPairStages = 8;
__host__ __device__ constexpr int kPairBoxRowsAt(int i) { return 16 * (i + 1); }

// ---------------------------------------------------------------- work map
// Tile plan of one expert with c > 0 rows and token tiles of at most bn rows
// (bn a multiple of 16): nt = ceil(c / tsz) tiles of tsz =
// roundup16(ceil(c / ceil(c / bn))) rows, so the tiles are balanced, every
// MMA-N is a multiple of 16 and tsz <= bn.  Returns (nt, tsz); (0, 1) for
// c <= 0.
__host__ __device__ inline int2 expert_tile_plan(int c, int bn) {
  if (c <= 0) return make_int2(0, 1);
  const int n0 = (c + bn - 1) / bn;
  const int tsz = (((c + n0 - 1) / n0) + 15) & ~15;
  return make_int2((c + tsz - 1) / tsz, tsz);
}

// Largest tile list the plan above gives R expanded rows over E experts with
// tiles of at most bn >= 16 rows: an expert with c rows gets at most
// ceil(c / bn) <= c / bn + 1 tiles, so R / bn + min(E, R) + 1 entries.
__host__ __device__ inline int64_t max_work_tiles(int64_t R, int64_t E, int64_t bn) {
  return R / bn + (E < R ? E : R) + 1;
}

// Whether entry (x = expert, y = first row, z = rows, w) of a work map is
// one a GEMM with token tiles of at most bn rows can run: an expert below E,
// 1..bn rows inside the R expanded rows, w == 0.  Written so that no sum can
// overflow, whatever the entry holds.
__host__ __device__ inline bool tile_entry_ok(int x, int y, int z, int w, int bn, int R, int E) {
  return x >= 0 && x < E && z >= 1 && z <= bn && y >= 0 && y <= R - z && w == 0;
}

// Activation encodings written by the expansion and h-quantisation kernels
// and read by the GEMMs:
//   kActFp8Row: E4M3 codes, one float scale per row (W4A8; the GEMM's weights
//               are E2M1);
//   kActMxfp8:  E4M3 codes, one E8M0 byte per 32 elements (W8A8; E4M3
//               weights);
//   kActSplit:  two MXFP8 terms per element -- hi, then the residual lo --
//               in rows of 2K codes (W4A16: bf16 activations on the FP8
//               tensor cores; E2M1 weights).
enum ActQuant : int { kActFp8Row = 0, kActMxfp8 = 1, kActSplit = 2 };

// MXFP8 and split activations: the (B operand) scale bytes are written by the
// quantisers straight into the GEMM's per-tile layout.  For tile t of the
// GEMM tile list and K stage ks there is one kSfbTileBytes block at
// (t * KS + ks) * kSfbTileBytes; tile row n's four scale bytes (K blocks
// 4ks .. 4ks+3) sit at sfb_row_offset(n): the 32-lane x 16-byte shape of the
// weight scale blocks, one 512-byte half per 128 rows.  Split activations
// (tiles of <= 128 rows): the hi term's bytes in the first half, the lo
// term's at the same offsets + kSfbLoOffset.
constexpr int kSfbTileBytes = 1024;   // up to 256 tile rows
constexpr int kSfbLoOffset = 512;     // the split's lo term
__host__ __device__ inline uint32_t sfb_row_offset(int n) {
  return static_cast<uint32_t>((n >> 7) * 512 + 16 * (n & 31) + 4 * ((n >> 5) & 3));
}
// Byte offset (K stage 0) of expanded row r's scales, from its expert's
// first row off_e and tile plan (first tile, rows per tile).
__host__ __device__ inline int64_t sfb_row_base(int r, int off_e, int2 plan, int KS) {
  const int j = r - off_e;
  const int q = j / plan.y;
  return (static_cast<int64_t>(plan.x) + q) * KS * kSfbTileBytes + sfb_row_offset(j - q * plan.y);
}

struct GemmArgs {
  const CUtensorMap* tmap_w;   // host copies, passed by value to the kernel
  const CUtensorMap* tmap_x;   // kNumXMaps maps, box heights kXBoxRows
  const CUtensorMap* tmap_sf;  // prepared scale blocks as uint32 [blocks, 128]
  const int4* tiles;           // (expert, first row, rows, 0)
  const int32_t* num_tiles;    // device scalar
  const float* row_scale;      // per-row activation scale
  void* out;                   // bf16 output
  int32_t m_per_expert;        // 2I (GEMM1) or H (GEMM2)
  int32_t k;                   // H (GEMM1) or I (GEMM2)
  int32_t out_ld;              // I (GEMM1) or H (GEMM2)
  int32_t* status;
  uint64_t timeout_ns;
  uint32_t a_tx_bytes;         // transaction bytes one weight TMA box counts
  int32_t num_sms;
  int32_t prefetch_stages;     // L2 prefetch distance of weight tiles, in K stages
  int32_t act;                 // ActQuant of the activations (and so the weights' type)
  const uint8_t* sfb_tiled;    // MXFP8 / split: activation scales in the per-tile layout
  const uint8_t* w_base;       // prepared weight boxes (for the optional L2 prefetcher)
  const CUtensorMap* tmap_x_pair;  // kNumXMaps maps, box heights kPairBoxRowsAt (or null)
  int32_t max_tiles;           // entries the tile list's allocation holds
  // The tile list was complete before the previous kernel passed its grid
  // wait, so the weight copies may start before this kernel's wait.
  bool early_list;
  // GEMM1 of W4A8 only, or null: the activations are token-major (gather_x:
  // [T, K] codes) and the kernel gathers each tile's rows by token (token =
  // gather_slot[row] / gather_k); see gemm_gather_supported.
  const int32_t* gather_slot;
  int32_t gather_k;
  const uint8_t* gather_x;
  // GEMM2 only, or null: the epilogue also forms the top-k combine (see
  // CombineArgs in gemm_common.cuh).
  int32_t* cmb_cnt;            // [T, m_per_expert / 128, 4] arrival counters, zero on entry
  const int32_t* cmb_slot;     // token_slot [R]
  const int32_t* cmb_row_of;   // row_of [T, k]
  const float* cmb_wts;        // routing weights [T, k]
  void* cmb_out;               // bf16 out [T, m_per_expert]
  int32_t cmb_k;
};

// zero / nzero (nullable): int32 words the kernel clears after its grid
// wait (the fused combine's counters).
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* wts,
                         int32_t* chunk_counts, int32_t* status, int32_t* zero, int64_t nzero,
                         cudaStream_t s);
// Activation outputs of the expansion kernels, by encoding.  kActFp8Row:
// FP8 codes xq [R, H] and x_scale (per-row float).  kActMxfp8: codes, x_sf
// (row-major scale bytes [R, H/32]) and sfb (per-tile layout above).
// kActSplit: codes [R, 2H], x_sf [R, 2H/32] and sfb.
struct QuantOut {
  uint8_t* xq;
  float* x_scale;
  int act;
  uint8_t* x_sf;
  uint8_t* sfb;
  // kActFp8Row with a staged x only: the codes of token t go to row t of xq
  // (token-major [T, H], which GEMM1 gathers rows from) instead of the k
  // expanded rows; x_scale is still written per expanded row.
  bool token_major;
};
// GEMM1 weights the tiny-batch front end asks L2 for: the first `boxes` K
// stages (prepared E2M1 boxes of kFp4BoxBytes, and their 512-byte scale
// blocks) of GEMM1's items 0 .. first_items-1 (the items its CTAs take
// first), from `ctas` extra CTAs.  Disabled when w is null or ctas == 0.
constexpr int kFp4BoxBytes = kTileM * kTileK / 2;
constexpr int kTinyPrefetchTiles = 160;   // tiles a prefetch CTA maps (>= the items of a round)
struct TinyPrefetch {
  const uint8_t* w;    // prepared w1 boxes
  const uint8_t* sf;   // prepared w1 scale blocks
  int32_t mt, ks;      // GEMM1's M-tiles per expert and K stages
  int32_t first_items;
  int32_t boxes;
  int32_t ctas;
};
cudaError_t launch_route_expand_tiny(const float* logits, const void* x, int T, int E, int k,
                                     int H, int bn, int32_t* ids, float* wts, int32_t* counts,
                                     int32_t* offsets, int4* tiles, int32_t* num_tiles,
                                     int2* tile_plan, int32_t* row_of, int32_t* token_slot,
                                     uint8_t* xq, float* x_scale, int32_t* status,
                                     const TinyPrefetch& pf, int32_t* zero, int64_t nzero,
                                     cudaStream_t s);
cudaError_t launch_expand_small(const void* x, const int32_t* ids, int T, int E, int k, int H,
                                int bn, int32_t* counts, int32_t* offsets, int4* tiles,
                                int32_t* num_tiles, int2* tile_plan, int32_t* row_of,
                                int32_t* token_slot, const QuantOut& q, cudaStream_t s);
// tile_plan (nullable): per expert (first tile, rows per tile).
// status (nullable): where a timed-out wait of the scan's bulk copies is
// recorded.
cudaError_t launch_scan(const int32_t* chunk_counts, int num_chunks, int E, int bn,
                        int32_t* counts, int32_t* offsets, int32_t* chunk_base, int4* tiles,
                        int32_t* num_tiles, int2* tile_plan, int32_t* status, cudaStream_t s);
cudaError_t launch_rank(const int32_t* ids, const int32_t* chunk_base, int T, int E, int k,
                        int32_t* row_of, int32_t* token_slot, cudaStream_t s);
// One CTA per token: the rows of its slots (from the per-chunk bases the
// scan leaves in chunk_base) into row_of / token_slot, and the token's
// quantised activations into them.
// x_on_device: x is device memory (else page-locked host memory read in
// place), which lets the kernel stage each token's row by a bulk copy.
// status: where a timed-out wait for that copy is recorded.
cudaError_t launch_quant_scatter(const void* x, bool x_on_device, const int32_t* chunk_base,
                                 const int32_t* ids, const int32_t* offsets, const int2* tile_plan,
                                 int T, int E, int k, int H, int32_t* row_of, int32_t* token_slot,
                                 const QuantOut& q, int32_t* status, cudaStream_t s);
// Per-row FP8 quantisation of h; status / timeout_ns: the bounded wait of
// its staged form.
cudaError_t launch_hquant(const void* h, int R, int I, uint8_t* hq, float* h_scale,
                          int32_t* status, uint64_t timeout_ns, cudaStream_t s);
// MXFP8 quantisation (act kActMxfp8) or two-term split (kActSplit) of h:
// codes, row-major scale bytes and the per-tile scale layout of GEMM2.
cudaError_t launch_hquant_mx(int act, const void* h, int R, int I, const int32_t* ids,
                             const int32_t* token_slot, const int32_t* offsets,
                             const int2* tile_plan, uint8_t* hq, uint8_t* h_sf, uint8_t* sfb,
                             int32_t* status, uint64_t timeout_ns, cudaStream_t s);
// status / timeout_ns: the bounded wait for the combine's staging copies.
cudaError_t launch_combine(const void* y, const float* wts, const int32_t* row_of, int T, int k,
                           int H, void* out, int32_t* status, uint64_t timeout_ns,
                           cudaStream_t s);
cudaError_t launch_gemm(bool swiglu, int variant, const GemmArgs& a, cudaStream_t s);
// Whether the W4A8 GEMM of tile variant 1..5 can gather token-major
// activation rows (its shared memory holds the producers' token lists).
bool gemm_gather_supported(int variant);
// The grouped GEMM on CTA pairs (gemm_pair.cu): W4A8 operands, M-tiles
// taken two at a time, so m_per_expert must be a multiple of 256; needs
// tmap_x_pair.
bool gemm_pair_supported(int m_per_expert, int act);
cudaError_t launch_gemm_pair(bool swiglu, const GemmArgs& a, cudaStream_t s);
// Tile variants 1..kMaxTileVariant; the largest token tile of each (the tile
// list is built with this bound).
constexpr int kMaxTileVariant = 6;
int gemm_tile_tokens(int variant, int act);
// Re-lays one weight tensor [E, M, K] (E2M1 with K/2 bytes per row, or E4M3
// with K bytes per row when fp8) and its scales [E, M, K/32] for the GEMM;
// swiglu_I > 0 applies GEMM1's gate/up row interleave (M = 2 * swiglu_I).
cudaError_t launch_prepare(const uint8_t* w, const uint8_t* sf, uint8_t* w_p, uint8_t* sf_p,
                           int E, int M, int K, int swiglu_I, bool fp8, cudaStream_t s);
// Sets the message moe_last_error() returns on the calling thread.
void set_last_error(const char* msg);
// The current device's check every entry point that launches kernels makes:
// MOE_OK on an sm_103a device (its SM count in *num_sms when not null), else
// MOE_ERR_UNSUPPORTED or MOE_ERR_CUDA with the message set.
int32_t check_device(int* num_sms);

cudaError_t launch_timeout_selftest(int32_t* status, uint64_t timeout_ns, cudaStream_t s);

}  // namespace moe
