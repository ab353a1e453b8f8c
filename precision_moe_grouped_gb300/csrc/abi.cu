// abi.cu -- the C ABI (include/moe.h): argument validation, workspace
// carving, TMA descriptor encoding and the launch sequence of the fused MoE
// forward.  Host code only; the kernels live in route.cu, gemm.cu, rowops.cu
// and prepare.cu.
//
// Pages cited (title and section):
//   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
//           MXFP4xFP8 CUTLASS MoE backend for SM90": Description (precomputed
//           grouped GEMM work scheduling and TMA descriptor state before the
//           GEMM launch), review comments (validate n % 16 / k % 64 and
//           K % 32 at the API boundary with clear errors; an empty routed
//           batch is a no-op).
//   [P4411] flashinfer PR #4411, "revert(moe): revert #3738 SM90 CUTLASS MoE
//           backend (+ dependents #4025, #4080) on release-v0.6.17":
//           Description (caller-owned workspace + size query; a null TMA
//           descriptor raised an illegal instruction that surfaced in a later
//           op).
//   [P3614] flashinfer PR #3614, "fix: make the cutlass MoE gemm profiler
//           MXFP8-aware": description (never launch with a null scale buffer;
//           fail fast at init instead of a deep kernel assert).
//
// Every pointer, size and alignment is checked here before the first CUDA
// call, and no tensor map is ever encoded from a null base address.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

thread_local char g_last_error[512] = "";

int32_t fail(int32_t code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int32_t fail(int32_t code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

#define MOE_CUDA(call)                                                                  \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(MOE_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));        \
  } while (0)

constexpr size_t kAlign = 256;

// A 128-row x 128-element E2M1 weight box copied with 16U4_ALIGN16B fills
// 16 KB of shared memory (8 data bytes + an 8-byte gap per 16 elements) but
// counts as the 8 KB of packed global bytes in the mbarrier transaction
// count (measured on GB300).
constexpr uint32_t kWeightBoxTxBytes = 128u * 128u / 2u;

// Default L2 prefetch distance of the GEMMs' weight stream (the prefetch
// warp), in fills: off.  It measured 15-25% slower on decode tiles and, once
// waiting warps sleep instead of spinning, neutral on prefill tiles (DSV3
// T=4096: 1797 us with a distance of 8, 1800 us without).
int default_prefetch(int) { return 0; }

// Tiny batches: CTAs the front end adds to ask L2 for GEMM1's first weight
// boxes, and the K stages it asks for per item (8, 16, 32 measured at DSV3
// T=1: 48.1, 47.7, 48.0 us).
constexpr int kTinyPrefetchCtas = 64;
constexpr int kTinyPrefetchBoxes = 16;

// Persistent-GEMM grid.  A tile holds at least one row, so a GEMM has at
// most T * k * m_tiles work items; with few rows per expert (T * k <= E / 4)
// tokens rarely share an expert and the bound is (nearly) the count -- exact
// at T = 1, whose k experts are distinct.  The grid is then the fewest CTAs
// that give every CTA the same number of rounds (DSV3 T=1 GEMM1: 256 items on
// 128 CTAs x 2 instead of 104 CTAs with 2 and 48 with 1), so no round runs on
// part of the GPU while the rest waits.  Otherwise one CTA per SM.
int gemm_grid(int num_sms, int64_t T, int k, int E, int m_tiles) {
  const int64_t rows = T * k;
  if (4 * rows > E) return num_sms;
  const int64_t items = rows * m_tiles;
  const int64_t rounds = (items + num_sms - 1) / num_sms;
  return static_cast<int>((items + rounds - 1) / rounds);
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int32_t check_shape(const moe_shape* s, int32_t mode) {
  if (!s) return fail(MOE_ERR_INVALID_ARG, "shape is NULL");
  if (mode < 0 || mode > 2) return fail(MOE_ERR_INVALID_ARG, "quant_mode %d unknown", mode);
  if (s->num_tokens < 0) return fail(MOE_ERR_INVALID_ARG, "num_tokens < 0");
  if (s->num_experts < 1 || s->num_experts > 1024)
    return fail(MOE_ERR_INVALID_ARG, "num_experts must be in [1, 1024]");
  if (s->top_k < 1 || s->top_k > s->num_experts || s->top_k > 32)
    return fail(MOE_ERR_INVALID_ARG, "top_k must be in [1, min(num_experts, 32)]");
  if (s->hidden <= 0 || s->inter <= 0) return fail(MOE_ERR_INVALID_ARG, "hidden/inter <= 0");
  if (s->hidden % 128 != 0 || s->inter % 128 != 0)
    return fail(MOE_ERR_MISALIGNED, "hidden (%d) and inter (%d) must be multiples of 128",
                s->hidden, s->inter);
  if (static_cast<int64_t>(s->num_tokens) * s->top_k >= (int64_t(1) << 31))
    return fail(MOE_ERR_INVALID_ARG, "num_tokens * top_k must be < 2^31");
  if (static_cast<int64_t>(s->num_experts) * 2 * s->inter >= (int64_t(1) << 31) ||
      static_cast<int64_t>(s->num_experts) * s->hidden >= (int64_t(1) << 31))
    return fail(MOE_ERR_INVALID_ARG, "num_experts * rows must be < 2^31");
  // The GEMMs address a weight box by its first row in one tensor map over
  // all experts' boxes, a 32-bit TMA coordinate: E * 2I * H / 128 rows for w1
  // (w2 has half as many).
  if (static_cast<int64_t>(s->num_experts) * 2 * s->inter * (s->hidden / 128) >=
      (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED,
                "num_experts * 2 * inter * hidden / 128 must be < 2^31 (32-bit weight-box "
                "row coordinates)");
  // A GEMM's work items (tiles x M-tiles) are counted in 32 bits: at most
  // (R / 16 + min(E, R) + 1) tiles times max(2I, H) / 128 M-tiles.
  {
    const int64_t R = static_cast<int64_t>(s->num_tokens) * s->top_k;
    const int64_t tiles = moe::max_work_tiles(R, s->num_experts, moe::kTinyBN);
    const int64_t mtiles = (2 * s->inter > s->hidden ? 2 * s->inter : s->hidden) / 128;
    if (tiles * mtiles >= (int64_t(1) << 31))
      return fail(MOE_ERR_UNSUPPORTED, "too many GEMM work items for 32-bit counters");
  }
  return MOE_OK;
}

// The activation encoding of a quantisation mode: per-row FP8 (W4A8),
// MXFP8 (W8A8), or the two-term MXFP8 split of the bf16 activations
// (W4A16).
int act_of(int32_t mode) {
  return mode == MOE_W8A8_MXFP8 ? moe::kActMxfp8
         : mode == MOE_W4A16_MXFP4_BF16 ? moe::kActSplit
                                         : moe::kActFp8Row;
}

void compute_layout(const moe_shape* s, int32_t mode, moe_ws_layout* L) {
  std::memset(L, 0, sizeof(*L));
  const int64_t T = s->num_tokens, E = s->num_experts, k = s->top_k, H = s->hidden,
                I = s->inter;
  const int64_t R = T * k;
  const int64_t chunks = (T + moe::kRouteChunk - 1) / moe::kRouteChunk;
  const int64_t max_tiles = moe::max_work_tiles(R, E, moe::kTinyBN);   // smallest tiles
  size_t off = 0;
  auto take = [&](int64_t bytes) {
    off = align_up(off, kAlign);
    const size_t o = off;
    off += static_cast<size_t>(bytes > 0 ? bytes : 0);
    return static_cast<uint64_t>(o);
  };
  L->status = take(16);
  L->ids = take(R * 4);
  L->weights = take(R * 4);
  L->row_of = take(R * 4);
  L->counts = take(E * 4);
  L->offsets = take((E + 1) * 4);
  L->chunk_counts = take(chunks * E * 4);
  L->token_slot = take(R * 4);
  L->tiles = take(max_tiles * 16);
  // W4A16: two FP8 terms per element (the split activations)
  const int act = act_of(mode);
  const int64_t terms = act == moe::kActSplit ? 2 : 1;
  L->xq = take(R * H * terms);
  L->x_scale = take(R * 4);
  L->h = take(R * I * 2);
  L->hq = take(R * I * terms);
  L->h_scale = take(R * 4);
  L->y = take(R * H * 2);
  L->x_stage = take(T * H * 2);
  L->logits_stage = take(T * E * 4);
  L->out_stage = take(T * H * 2);
  L->tile_plan = take(E * 8);
  // MXFP8 / split activation scales: row-major bytes and the GEMMs' per-tile
  // layout
  const bool mx = act != moe::kActFp8Row;
  L->x_sf = take(mx ? R * (H / 32) * terms : 0);
  L->h_sf = take(mx ? R * (I / 32) * terms : 0);
  L->x_sf_tiled = take(mx ? max_tiles * (H / 128) * moe::kSfbTileBytes : 0);
  L->h_sf_tiled = take(mx ? max_tiles * (I / 128) * moe::kSfbTileBytes : 0);
  // last: the fused combine's arrival counters [T, H/128, 4] (at
  // combine_cnt_offset)
  take(T * (H / 128) * 4 * 4);
  L->total = align_up(off, kAlign);
  L->max_tiles = static_cast<int32_t>(max_tiles);
  L->num_chunks = static_cast<int32_t>(chunks);
}

// The fused combine's counters: the workspace's last region.
uint64_t combine_cnt_offset(const moe_shape* s, const moe_ws_layout& L) {
  const uint64_t bytes = static_cast<uint64_t>(s->num_tokens) * (s->hidden / 128) * 16;
  return L.total - align_up(bytes, kAlign);
}

// ----------------------------------------------------------- device state
struct DeviceInfo {
  int num_sms = 0;
  bool ok = false;
};

int32_t device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(MOE_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev].ok) {
    int major = 0, minor = 0, sms = 0;
    MOE_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    MOE_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    MOE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (major != 10 || minor != 3)
      return fail(MOE_ERR_UNSUPPORTED,
                  "this library is built for sm_103a (GB300); device %d is sm_%d%d", dev, major,
                  minor);
    cache[dev].num_sms = sms;
    cache[dev].ok = true;
  }
  *out = cache[dev];
  return MOE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

enum class MapKind { kFp4Weights, kBytes, kScaleBlocks };

// 2-D tensor map over a row-major [rows, cols] matrix of `kind` elements;
// box = box_cols x box_rows elements.
//   kFp4Weights:  E2M1 codes, 16U4_ALIGN16B (each group of 16 packed codes
//                 lands as 16 bytes in shared memory), 128-byte swizzle
//   kBytes:       uint8 (FP8 codes), 128-byte swizzle
//   kScaleBlocks: uint32 words, no swizzle
int32_t make_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, MapKind kind,
                  uint32_t box_cols, uint32_t box_rows) {
  if (!base) return fail(MOE_ERR_INVALID_ARG, "refusing to encode a tensor map for NULL");
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const bool fp4 = kind == MapKind::kFp4Weights, words = kind == MapKind::kScaleBlocks;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {fp4 ? cols / 2 : words ? cols * 4 : cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m,
                  fp4     ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B
                  : words ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                          : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  words ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) rows=%llu cols=%llu kind=%d",
                static_cast<int>(r), static_cast<unsigned long long>(rows),
                static_cast<unsigned long long>(cols), static_cast<int>(kind));
  return MOE_OK;
}

int pick_variant(const moe_shape* s, const moe_options* o) {
  if (o && o->tile_variant >= 1 && o->tile_variant <= moe::kMaxTileVariant) return o->tile_variant;
  const double rows_per_expert =
      static_cast<double>(s->num_tokens) * s->top_k / static_cast<double>(s->num_experts);
  // Measured on the DSV3 shape (T = 64 .. 4096): 16-token tiles (12 stages)
  // are fastest while experts average <= 8 rows; 32-token tiles (10 stages)
  // up to 32 rows (T=1024: 1.27 ms against 1.35 ms for 160-token tiles);
  // from 48 rows on the 6-stage 160-token tiles (T=1536: 1.39 ms against
  // 1.63 ms), which also beat 5-stage 224-token tiles at T=4096.
  return rows_per_expert <= 8.0 ? 3 : rows_per_expert <= 32.0 ? 1 : 5;
}

int32_t check_options(const moe_options* o) {
  if (!o) return MOE_OK;
  if (o->tile_variant < 0 || o->tile_variant > moe::kMaxTileVariant)
    return fail(MOE_ERR_INVALID_ARG, "tile_variant must be in [0, %d]", moe::kMaxTileVariant);
  if (o->timeout_ms < 0) return fail(MOE_ERR_INVALID_ARG, "timeout_ms < 0");
  if (o->prefetch_stages > 1024) return fail(MOE_ERR_INVALID_ARG, "prefetch_stages > 1024");
  if (o->gather_x < -1 || o->gather_x > 1)
    return fail(MOE_ERR_INVALID_ARG, "gather_x must be -1, 0 or 1");
  if (o->fuse_combine < -1 || o->fuse_combine > 1)
    return fail(MOE_ERR_INVALID_ARG, "fuse_combine must be -1, 0 or 1");
  if (o->reserved[0] != 0) return fail(MOE_ERR_INVALID_ARG, "reserved option fields must be 0");
  return MOE_OK;
}

int32_t check_forward_args(const moe_shape* shape, int32_t mode, const void* x,
                           const float* logits, const void* w1, const void* w1_sf,
                           const void* w2, const void* w2_sf, const void* out, void* ws,
                           size_t ws_bytes, const moe_options* opts) {
  int32_t st = check_shape(shape, mode);
  if (st != MOE_OK) return st;
  if ((st = check_options(opts)) != MOE_OK) return st;
  if (shape->num_tokens == 0) return MOE_OK;
  if (!x || !logits || !w1 || !w1_sf || !w2 || !w2_sf || !out || !ws)
    return fail(MOE_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(logits, 4))
    return fail(MOE_ERR_MISALIGNED, "x/out must be 16-byte aligned, logits 4-byte aligned");
  if (!aligned(w1, 256) || !aligned(w2, 256) || !aligned(w1_sf, 256) || !aligned(w2_sf, 256) ||
      !aligned(ws, 256))
    return fail(MOE_ERR_MISALIGNED, "weights, scales and workspace must be 256-byte aligned");
  moe_ws_layout L;
  compute_layout(shape, mode, &L);
  if (ws_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < required %llu", ws_bytes,
                static_cast<unsigned long long>(L.total));
  return MOE_OK;
}

template <typename T>
T* at(void* ws, uint64_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// The address under which this device's kernels reach host buffer p in
// place: page-locked host memory (cudaHostAlloc, cudaMallocHost,
// cudaHostRegister), which unified addressing maps into every device --
// else nullptr (pageable memory, or memory of another device): the caller
// then stages the buffer with copies.
const void* host_in_place(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();   // clear the sticky-free error of an unknown pointer
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Whether p is device memory of the current device (cudaMalloc), which
// bulk copies may read; host-mapped and unregistered pointers are not.
bool on_device(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int dev = -1;
  return a.type == cudaMemoryTypeDevice && cudaGetDevice(&dev) == cudaSuccess && a.device == dev;
}

// x_on_device: x is device memory (see on_device).
int32_t run_forward(const moe_shape* s, int32_t mode, const void* x, const float* logits,
                    const void* w1, const void* w1_sf, const void* w2, const void* w2_sf,
                    void* out, void* ws, cudaStream_t st, const moe_options* opts,
                    bool x_on_device) {
  DeviceInfo dev;
  int32_t rc = device_info(&dev);
  if (rc != MOE_OK) return rc;
  moe_ws_layout L;
  compute_layout(s, mode, &L);
  const int act = act_of(mode);
  const bool fp8w = act == moe::kActMxfp8;       // E4M3 weights (else E2M1)
  const bool tiled = act != moe::kActFp8Row;     // per-32 activation scales
  const int T = s->num_tokens, E = s->num_experts, k = s->top_k, H = s->hidden, I = s->inter;
  const int R = T * k;
  const int terms = act == moe::kActSplit ? 2 : 1;
  const int variant = pick_variant(s, opts);
  const int bn = moe::gemm_tile_tokens(variant, act);
  const int prefetch = !opts || opts->prefetch_stages == 0 ? default_prefetch(variant)
                       : opts->prefetch_stages < 0 ? 0 : opts->prefetch_stages;
  const uint64_t timeout_ns =
      static_cast<uint64_t>(opts && opts->timeout_ms > 0 ? opts->timeout_ms : 1000) * 1000000ull;
  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* num_tiles = status + 1;
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* wts = at<float>(ws, L.weights);
  int32_t* row_of = at<int32_t>(ws, L.row_of);
  int32_t* chunk = at<int32_t>(ws, L.chunk_counts);
  int4* tiles = at<int4>(ws, L.tiles);
  uint8_t* xq = at<uint8_t>(ws, L.xq);
  float* x_scale = at<float>(ws, L.x_scale);
  void* h = at<void>(ws, L.h);
  uint8_t* hq = at<uint8_t>(ws, L.hq);
  float* h_scale = at<float>(ws, L.h_scale);
  void* y = at<void>(ws, L.y);
  int2* tile_plan = at<int2>(ws, L.tile_plan);
  uint8_t* x_sf = tiled ? at<uint8_t>(ws, L.x_sf) : nullptr;
  uint8_t* h_sf = tiled ? at<uint8_t>(ws, L.h_sf) : nullptr;
  uint8_t* sfb1 = tiled ? at<uint8_t>(ws, L.x_sf_tiled) : nullptr;
  uint8_t* sfb2 = tiled ? at<uint8_t>(ws, L.h_sf_tiled) : nullptr;

  CUtensorMap tm_w1, tm_w2, tm_sf1, tm_sf2, tm_x[moe::kNumXMaps], tm_h[moe::kNumXMaps];
  CUtensorMap tm_xp[moe::kNumXMaps], tm_hp[moe::kNumXMaps];   // CTA-pair half boxes
  // prepared weights: contiguous 128-row x 128-element boxes (64-byte rows
  // of E2M1 codes, or 128-byte rows of E4M3 codes in MXFP8); prepared
  // scales: one 512-byte block per box
  const uint64_t w1_boxes = static_cast<uint64_t>(E) * (2 * I / 128) * (H / 128);
  const uint64_t w2_boxes = static_cast<uint64_t>(E) * (H / 128) * (I / 128);
  const MapKind wkind = fp8w ? MapKind::kBytes : MapKind::kFp4Weights;
  const uint32_t w_tx = fp8w ? 128u * 128u : kWeightBoxTxBytes;
  if ((rc = make_tmap(&tm_w1, w1, w1_boxes * 128, 128, wkind, 128, 128)) != MOE_OK ||
      (rc = make_tmap(&tm_w2, w2, w2_boxes * 128, 128, wkind, 128, 128)) != MOE_OK ||
      (rc = make_tmap(&tm_sf1, w1_sf, w1_boxes, 128, MapKind::kScaleBlocks, 128, 1)) != MOE_OK ||
      (rc = make_tmap(&tm_sf2, w2_sf, w2_boxes, 128, MapKind::kScaleBlocks, 128, 1)) != MOE_OK)
    return rc;
  for (int i = 0; i < moe::kNumXMaps; ++i) {
    const uint32_t rows = static_cast<uint32_t>(moe::kXBoxRowsAt(i));
    // split activations: rows of 2K codes (hi terms, then lo terms)
    if ((rc = make_tmap(&tm_x[i], xq, R, static_cast<uint64_t>(terms) * H, MapKind::kBytes, 128,
                        rows)) != MOE_OK ||
        (rc = make_tmap(&tm_h[i], hq, R, static_cast<uint64_t>(terms) * I, MapKind::kBytes, 128,
                        rows)) != MOE_OK)
      return rc;
  }
  const bool pair = variant == 6 && mode == MOE_W4A8_MXFP4_FP8;
  if (pair)
    for (int i = 0; i < moe::kNumXMaps; ++i) {
      const uint32_t rows = static_cast<uint32_t>(moe::kPairBoxRowsAt(i));
      if ((rc = make_tmap(&tm_xp[i], xq, R, H, MapKind::kBytes, 128, rows)) != MOE_OK ||
          (rc = make_tmap(&tm_hp[i], hq, R, I, MapKind::kBytes, 128, rows)) != MOE_OK)
        return rc;
    }

  cudaEvent_t* ev = opts ? static_cast<cudaEvent_t*>(opts->stage_events) : nullptr;
  int stage = 0;
  auto mark = [&]() -> cudaError_t {
    return ev ? cudaEventRecord(ev[stage++], st) : cudaSuccess;
  };
  const int grid1 = gemm_grid(dev.num_sms, T, k, E, 2 * I / moe::kTileM);
  const int grid2 = gemm_grid(dev.num_sms, T, k, E, H / moe::kTileM);
  // the first kernel clears the status word; tiny batches (W4A8) route,
  // expand and quantise in one kernel, small batches expand in one kernel
  // GEMM1 gathers token-major activation rows (W4A8 large batches with x on
  // the device, staged by the expansion; not on CTA pairs)
  const bool large = !(T <= moe::kTinyT && mode == MOE_W4A8_MXFP4_FP8) && T > moe::kSmallT;
  const bool gather = opts && opts->gather_x > 0 && mode == MOE_W4A8_MXFP4_FP8 && large &&
                      x_on_device && H * 2 <= 48 * 1024 && moe::gemm_gather_supported(variant);
  const moe::QuantOut qx{xq, x_scale, act, x_sf, sfb1, gather};
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* token_slot = at<int32_t>(ws, L.token_slot);
  // GEMM2's epilogue forms the combine (one-CTA kernel); the front end
  // clears its counters
  const bool fuse_cmb = opts && opts->fuse_combine > 0 && variant != 6;
  int32_t* cmb_cnt = fuse_cmb ? at<int32_t>(ws, combine_cnt_offset(s, L)) : nullptr;
  const int64_t cmb_n = static_cast<int64_t>(T) * (H / moe::kTileM) * 4;
  MOE_CUDA(mark());
  // large batches: the scan writes the tile list, the scatter kernel follows
  const bool large_front = large;
  if (T <= moe::kTinyT && mode == MOE_W4A8_MXFP4_FP8) {
    // extra CTAs of the front end start GEMM1's weight stream into L2: the
    // first kTinyPrefetchBoxes K stages of the items GEMM1's CTAs take
    // first -- when those are a large share of all items (at most two
    // rounds of the grid: DSV3 T=1 48.6 -> 47.7 us; at T=8, a dozen rounds,
    // it measured 1.4 us slower)
    const int64_t items_max = static_cast<int64_t>(R) * (2 * I / moe::kTileM);
    const bool prefetch_w1 = items_max <= 2 * static_cast<int64_t>(grid1);
    const moe::TinyPrefetch pf{static_cast<const uint8_t*>(w1), static_cast<const uint8_t*>(w1_sf),
                               2 * I / moe::kTileM, H / moe::kTileK, grid1, kTinyPrefetchBoxes,
                               prefetch_w1 ? kTinyPrefetchCtas : 0};
    MOE_CUDA(moe::launch_route_expand_tiny(logits, x, T, E, k, H, bn, ids, wts,
                                           at<int32_t>(ws, L.counts), offsets, tiles, num_tiles,
                                           tile_plan, row_of, token_slot, xq, x_scale, status, pf,
                                           cmb_cnt, cmb_n, st));
    MOE_CUDA(mark());
    MOE_CUDA(mark());
    MOE_CUDA(mark());
    MOE_CUDA(mark());
  } else if (T <= moe::kSmallT) {
    MOE_CUDA(moe::launch_route(logits, T, E, k, ids, wts, chunk, status, cmb_cnt, cmb_n, st));
    MOE_CUDA(mark());
    MOE_CUDA(moe::launch_expand_small(x, ids, T, E, k, H, bn, at<int32_t>(ws, L.counts), offsets,
                                      tiles, num_tiles, tile_plan, row_of, token_slot, qx, st));
    MOE_CUDA(mark());
    MOE_CUDA(mark());
    MOE_CUDA(mark());
  } else {
    MOE_CUDA(moe::launch_route(logits, T, E, k, ids, wts, chunk, status, cmb_cnt, cmb_n, st));
    MOE_CUDA(mark());
    MOE_CUDA(moe::launch_scan(chunk, L.num_chunks, E, bn, at<int32_t>(ws, L.counts), offsets,
                              chunk, tiles, num_tiles, tile_plan, status, st));
    MOE_CUDA(mark());
    MOE_CUDA(mark());   // the scatter kernel ranks the rows itself (no rank kernel)
    MOE_CUDA(moe::launch_quant_scatter(x, x_on_device, chunk, ids, offsets, tile_plan, T, E, k,
                                       H, row_of, token_slot, qx, status, st));
    MOE_CUDA(mark());
  }
  // W4A8: the per-row token scale is applied in the epilogues; MXFP8 and
  // split: the block scales ride with the operands into the MMA
  moe::GemmArgs g1{&tm_w1, tm_x, &tm_sf1, tiles, num_tiles,
                   tiled ? nullptr : x_scale, h, 2 * I, H, I, status, timeout_ns, w_tx, grid1,
                   prefetch, act, sfb1, static_cast<const uint8_t*>(w1), pair ? tm_xp : nullptr,
                   L.max_tiles, large_front, gather ? token_slot : nullptr, k,
                   gather ? xq : nullptr};
  MOE_CUDA(moe::launch_gemm(true, variant, g1, st));
  MOE_CUDA(mark());
  if (tiled)
    MOE_CUDA(moe::launch_hquant_mx(act, h, R, I, ids, token_slot, offsets, tile_plan, hq, h_sf,
                                   sfb2, status, timeout_ns, st));
  else
    MOE_CUDA(moe::launch_hquant(h, R, I, hq, h_scale, status, timeout_ns, st));
  MOE_CUDA(mark());
  moe::GemmArgs g2{&tm_w2, tm_h, &tm_sf2, tiles, num_tiles,
                   tiled ? nullptr : h_scale, y, H, I, H, status, timeout_ns, w_tx, grid2,
                   prefetch, act, sfb2, static_cast<const uint8_t*>(w2), pair ? tm_hp : nullptr,
                   L.max_tiles, true, nullptr, 0, nullptr, cmb_cnt, token_slot, row_of, wts,
                   fuse_cmb ? out : nullptr, k};
  MOE_CUDA(moe::launch_gemm(false, variant, g2, st));
  MOE_CUDA(mark());
  if (!fuse_cmb)
    MOE_CUDA(moe::launch_combine(y, wts, row_of, T, k, H, out, status, timeout_ns, st));
  MOE_CUDA(mark());
  return MOE_OK;
}

}  // namespace

namespace moe {
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

int32_t check_device(int* num_sms) {
  DeviceInfo dev;
  const int32_t rc = device_info(&dev);
  if (rc == MOE_OK && num_sms) *num_sms = dev.num_sms;
  return rc;
}
}  // namespace moe

extern "C" {

const char* moe_version(void) { return "precision_moe_grouped_gb300 0.1 (sm_103a)"; }

const char* moe_last_error(void) { return g_last_error; }

const char* moe_stage_name(int32_t stage) {
  static const char* names[MOE_NUM_STAGES] = {"route", "scan", "rank", "quant_scatter",
                                              "gemm1", "hquant", "gemm2", "combine"};
  return stage >= 0 && stage < MOE_NUM_STAGES ? names[stage] : nullptr;
}

const char* moe_status_string(int32_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_MISALIGNED: return "misaligned pointer or shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side bounds check failed (checked build)";
    default: return "unknown status";
  }
}

size_t moe_workspace_size(const moe_shape* shape, int32_t quant_mode) {
  if (check_shape(shape, quant_mode) != MOE_OK) return 0;
  moe_ws_layout L;
  compute_layout(shape, quant_mode, &L);
  return static_cast<size_t>(L.total);
}

int32_t moe_workspace_layout(const moe_shape* shape, int32_t quant_mode, moe_ws_layout* layout) {
  int32_t st = check_shape(shape, quant_mode);
  if (st != MOE_OK) return st;
  if (!layout) return fail(MOE_ERR_INVALID_ARG, "layout is NULL");
  compute_layout(shape, quant_mode, layout);
  return MOE_OK;
}

int32_t moe_prepare_weights(const moe_shape* shape, int32_t quant_mode, const void* w1,
                            const void* w1_sf, const void* w2, const void* w2_sf, void* w1_p,
                            void* w1_sf_p, void* w2_p, void* w2_sf_p, void* stream) {
  int32_t st = check_shape(shape, quant_mode);
  if (st != MOE_OK) return st;
  const bool fp8 = quant_mode == MOE_W8A8_MXFP8;
  const void* ins[4] = {w1, w1_sf, w2, w2_sf};
  const void* outs[4] = {w1_p, w1_sf_p, w2_p, w2_sf_p};
  for (int i = 0; i < 4; ++i) {
    if (!ins[i] || !outs[i]) return fail(MOE_ERR_INVALID_ARG, "a weight pointer is NULL");
    if (!aligned(ins[i], 256) || !aligned(outs[i], 256))
      return fail(MOE_ERR_MISALIGNED, "weight buffers must be 256-byte aligned");
    if (ins[i] == outs[i]) return fail(MOE_ERR_INVALID_ARG, "prepared weights must not alias");
  }
  DeviceInfo dev;
  if ((st = device_info(&dev)) != MOE_OK) return st;
  const int E = shape->num_experts, H = shape->hidden, I = shape->inter;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_CUDA(moe::launch_prepare(static_cast<const uint8_t*>(w1), static_cast<const uint8_t*>(w1_sf),
                               static_cast<uint8_t*>(w1_p), static_cast<uint8_t*>(w1_sf_p), E,
                               2 * I, H, I, fp8, s));
  MOE_CUDA(moe::launch_prepare(static_cast<const uint8_t*>(w2), static_cast<const uint8_t*>(w2_sf),
                               static_cast<uint8_t*>(w2_p), static_cast<uint8_t*>(w2_sf_p), E, H,
                               I, 0, fp8, s));
  return MOE_OK;
}

int32_t moe_forward_ex(const moe_shape* shape, int32_t quant_mode, const void* x,
                       const float* router_logits, const void* w1_p, const void* w1_sf_p,
                       const void* w2_p, const void* w2_sf_p, void* out, void* workspace,
                       size_t workspace_bytes, void* stream, const moe_options* opts) {
  int32_t st = check_forward_args(shape, quant_mode, x, router_logits, w1_p, w1_sf_p, w2_p,
                                  w2_sf_p, out, workspace, workspace_bytes, opts);
  if (st != MOE_OK || shape->num_tokens == 0) return st;
  return run_forward(shape, quant_mode, x, router_logits, w1_p, w1_sf_p, w2_p, w2_sf_p, out,
                     workspace, static_cast<cudaStream_t>(stream), opts, on_device(x));
}

int32_t moe_forward(const moe_shape* shape, int32_t quant_mode, const void* x,
                    const float* router_logits, const void* w1_p, const void* w1_sf_p,
                    const void* w2_p, const void* w2_sf_p, void* out, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return moe_forward_ex(shape, quant_mode, x, router_logits, w1_p, w1_sf_p, w2_p, w2_sf_p, out,
                        workspace, workspace_bytes, stream, nullptr);
}

int32_t moe_forward_host(const moe_shape* shape, int32_t quant_mode, const void* x_host,
                         const float* logits_host, const void* w1_p, const void* w1_sf_p,
                         const void* w2_p, const void* w2_sf_p, void* out_host,
                         void* workspace, size_t workspace_bytes, void* stream,
                         const moe_options* opts) {
  int32_t st = check_shape(shape, quant_mode);
  if (st != MOE_OK) return st;
  if (shape->num_tokens == 0) return MOE_OK;
  if (!x_host || !logits_host || !out_host || !workspace)
    return fail(MOE_ERR_INVALID_ARG, "a required pointer is NULL");
  moe_ws_layout L;
  compute_layout(shape, quant_mode, &L);
  // Page-locked host buffers are read and written in place by the kernels
  // (over the host link); the others are staged through the workspace.
  const void* xd = host_in_place(x_host);
  const float* ld = static_cast<const float*>(host_in_place(logits_host));
  void* od = const_cast<void*>(host_in_place(out_host));
  const void* xin = xd ? xd : at<void>(workspace, L.x_stage);
  const float* lin = ld ? ld : at<float>(workspace, L.logits_stage);
  void* oout = od ? od : at<void>(workspace, L.out_stage);
  st = check_forward_args(shape, quant_mode, xin, lin, w1_p, w1_sf_p, w2_p, w2_sf_p, oout,
                          workspace, workspace_bytes, opts);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t T = shape->num_tokens, H = shape->hidden, E = shape->num_experts;
  if (!xd)
    MOE_CUDA(cudaMemcpyAsync(const_cast<void*>(xin), x_host, T * H * 2, cudaMemcpyHostToDevice,
                             s));
  if (!ld)
    MOE_CUDA(cudaMemcpyAsync(const_cast<float*>(lin), logits_host, T * E * 4,
                             cudaMemcpyHostToDevice, s));
  st = run_forward(shape, quant_mode, xin, lin, w1_p, w1_sf_p, w2_p, w2_sf_p, oout, workspace, s,
                   opts, xd == nullptr);
  if (st != MOE_OK) return st;
  if (!od) MOE_CUDA(cudaMemcpyAsync(out_host, oout, T * H * 2, cudaMemcpyDeviceToHost, s));
  return MOE_OK;
}

namespace {

// moe_forward_host_steps: the second staging set, after moe_forward's
// workspace (the first is the workspace's own x_stage / logits_stage /
// out_stage).
struct StepsLayout {
  uint64_t x, logits, out, end;
};

StepsLayout steps_layout(const moe_shape* s, const moe_ws_layout& L) {
  const uint64_t T = static_cast<uint64_t>(s->num_tokens), H = static_cast<uint64_t>(s->hidden),
                 E = static_cast<uint64_t>(s->num_experts);
  StepsLayout r;
  uint64_t off = L.total;
  r.x = off;
  off = align_up(off + T * H * 2, kAlign);
  r.logits = off;
  off = align_up(off + T * E * 4, kAlign);
  r.out = off;
  r.end = align_up(off + T * H * 2, kAlign);
  return r;
}

// The copy streams and events of one moe_forward_host_steps call; released
// when the call returns (the runtime defers the release until the work
// queued on them has finished).
struct StepsSync {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, in_ready[2] = {}, consumed[2] = {}, out_free[2] = {};
  cudaError_t create() {
    cudaError_t e = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&start, &in_ready[0], &in_ready[1], &consumed[0], &consumed[1],
                            &out_free[0], &out_free[1]})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    return e;
  }
  ~StepsSync() {
    for (cudaEvent_t ev : {start, in_ready[0], in_ready[1], consumed[0], consumed[1], out_free[0],
                           out_free[1]})
      if (ev) cudaEventDestroy(ev);
    if (h2d) cudaStreamDestroy(h2d);
    if (d2h) cudaStreamDestroy(d2h);
  }
};

}  // namespace

size_t moe_steps_workspace_size(const moe_shape* shape, int32_t quant_mode) {
  if (check_shape(shape, quant_mode) != MOE_OK) return 0;
  moe_ws_layout L;
  compute_layout(shape, quant_mode, &L);
  return static_cast<size_t>(steps_layout(shape, L).end);
}

int32_t moe_forward_host_steps(const moe_shape* shape, int32_t quant_mode, int32_t n_steps,
                               const void* const* x_host, const float* const* logits_host,
                               const void* w1_p, const void* w1_sf_p, const void* w2_p,
                               const void* w2_sf_p, void* const* out_host, void* workspace,
                               size_t workspace_bytes, void* stream, const moe_options* opts) {
  int32_t st = check_shape(shape, quant_mode);
  if (st != MOE_OK) return st;
  if (n_steps < 0) return fail(MOE_ERR_INVALID_ARG, "n_steps < 0");
  if (opts && opts->stage_events)
    return fail(MOE_ERR_INVALID_ARG, "stage_events is not supported over several steps");
  if (shape->num_tokens == 0 || n_steps == 0) return MOE_OK;
  if (!x_host || !logits_host || !out_host || !workspace)
    return fail(MOE_ERR_INVALID_ARG, "a required pointer is NULL");
  for (int32_t i = 0; i < n_steps; ++i)
    if (!x_host[i] || !logits_host[i] || !out_host[i])
      return fail(MOE_ERR_INVALID_ARG, "host buffer pointer of step %d is NULL", i);
  moe_ws_layout L;
  compute_layout(shape, quant_mode, &L);
  const StepsLayout S = steps_layout(shape, L);
  if (workspace_bytes < S.end)
    return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < required %llu",
                workspace_bytes, static_cast<unsigned long long>(S.end));
  void* const xs[2] = {at<void>(workspace, L.x_stage), at<void>(workspace, S.x)};
  float* const ls[2] = {at<float>(workspace, L.logits_stage), at<float>(workspace, S.logits)};
  void* const os[2] = {at<void>(workspace, L.out_stage), at<void>(workspace, S.out)};
  st = check_forward_args(shape, quant_mode, xs[0], ls[0], w1_p, w1_sf_p, w2_p, w2_sf_p, os[0],
                          workspace, workspace_bytes, opts);
  if (st != MOE_OK) return st;
  const size_t T = shape->num_tokens, H = shape->hidden, E = shape->num_experts;
  const size_t xb = T * H * 2, lb = T * E * 4, ob = T * H * 2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StepsSync q;
  MOE_CUDA(q.create());
  // the copy streams start after the work already queued on `stream`
  MOE_CUDA(cudaEventRecord(q.start, s));
  MOE_CUDA(cudaStreamWaitEvent(q.h2d, q.start, 0));
  MOE_CUDA(cudaStreamWaitEvent(q.d2h, q.start, 0));
  for (int32_t i = 0; i < n_steps; ++i) {
    const int b = i & 1;
    // staging set b: its inputs were consumed by step i - 2 (recorded after
    // that forward), its output copied out by step i - 2's D2H
    if (i >= 2) MOE_CUDA(cudaStreamWaitEvent(q.h2d, q.consumed[b], 0));
    MOE_CUDA(cudaMemcpyAsync(xs[b], x_host[i], xb, cudaMemcpyHostToDevice, q.h2d));
    MOE_CUDA(cudaMemcpyAsync(ls[b], logits_host[i], lb, cudaMemcpyHostToDevice, q.h2d));
    MOE_CUDA(cudaEventRecord(q.in_ready[b], q.h2d));
    MOE_CUDA(cudaStreamWaitEvent(s, q.in_ready[b], 0));
    if (i >= 2) MOE_CUDA(cudaStreamWaitEvent(s, q.out_free[b], 0));
    st = run_forward(shape, quant_mode, xs[b], ls[b], w1_p, w1_sf_p, w2_p, w2_sf_p, os[b],
                     workspace, s, opts, true);
    if (st != MOE_OK) return st;
    MOE_CUDA(cudaEventRecord(q.consumed[b], s));
    MOE_CUDA(cudaStreamWaitEvent(q.d2h, q.consumed[b], 0));
    MOE_CUDA(cudaMemcpyAsync(out_host[i], os[b], ob, cudaMemcpyDeviceToHost, q.d2h));
    MOE_CUDA(cudaEventRecord(q.out_free[b], q.d2h));
  }
  // `stream` reaches its end once every output has reached the host
  MOE_CUDA(cudaStreamWaitEvent(s, q.out_free[(n_steps - 1) & 1], 0));
  if (n_steps >= 2) MOE_CUDA(cudaStreamWaitEvent(s, q.out_free[n_steps & 1], 0));
  return MOE_OK;
}

int32_t moe_read_device_status(const void* workspace, void* stream, int32_t* status) {
  if (!workspace || !status) return fail(MOE_ERR_INVALID_ARG, "NULL workspace or status");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  MOE_CUDA(cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  *status = v;
  return MOE_OK;
}

int32_t moe_selftest_timeout(void* workspace, int32_t timeout_us, void* stream) {
  if (!workspace || !aligned(workspace, 256))
    return fail(MOE_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
  if (timeout_us <= 0 || timeout_us > 2000000)
    return fail(MOE_ERR_INVALID_ARG, "timeout_us must be in (0, 2e6]");
  DeviceInfo dev;
  int32_t st = device_info(&dev);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaMemsetAsync(workspace, 0, 16, s));
  MOE_CUDA(moe::launch_timeout_selftest(static_cast<int32_t*>(workspace),
                                        static_cast<uint64_t>(timeout_us) * 1000ull, s));
  return MOE_OK;
}

}  // extern "C"
