// noalloc.cu -- moe_route_noalloc: the routing front end of the forward
// (top-k routing, per-expert offsets, expert-major row map) for callers that
// cannot allocate device memory.
//
// Its scratch (the per-chunk expert histogram, per-expert counts, the row ->
// (token, slot) map and the GEMM tile list the scan kernel also writes) lives
// in one file-scope device array instead of a caller workspace.  The array
// is part of the library image: every GPU that loads the library holds it
// until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

__device__ __align__(256) uint8_t g_route_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Contexts whose scratch address is cached (further ones replace entries).
constexpr int kMaxContexts = 64;

// Records the message where moe_last_error() reads it and returns `code`.
int32_t noalloc_fail(int32_t code, const char* fmt, ...) {
  char msg[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof(msg), fmt, ap);
  va_end(ap);
  moe::set_last_error(msg);
  return code;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// Scratch carving for one call (offsets from the array's base).
struct Carve {
  size_t chunk_counts, counts, token_slot, tiles, num_tiles, total;
};

Carve carve(int64_t T, int64_t E, int64_t k) {
  const int64_t R = T * k;
  const int64_t chunks = (T + moe::kRouteChunk - 1) / moe::kRouteChunk;
  const int64_t max_tiles = moe::max_work_tiles(R, E, moe::kDecodeBN);
  Carve c{};
  size_t off = 0;
  c.chunk_counts = off;
  off = up256(off + static_cast<size_t>(chunks * E * 4));
  c.counts = off;
  off = up256(off + static_cast<size_t>(E * 4));
  c.token_slot = off;
  off = up256(off + static_cast<size_t>(R * 4));
  c.tiles = off;
  off = up256(off + static_cast<size_t>(max_tiles * 16));
  c.num_tiles = off;
  off = up256(off + 16);
  c.total = off;
  return c;
}

// Driver entry points for the current context and its process-unique id,
// looked up once through the runtime (the library links only cudart).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// Process-unique id of the calling thread's current context (0 if none).
int32_t current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  if (!get_current || !get_id)
    return noalloc_fail(MOE_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId entry points unavailable");
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS)
    return noalloc_fail(MOE_ERR_CUDA, "cuCtxGetCurrent failed");
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS)
    return noalloc_fail(MOE_ERR_CUDA, "cuCtxGetId failed");
  return MOE_OK;
}

// Device address of g_route_scratch in the calling thread's current CUDA
// context, looked up once per context with that context current and cached
// under the context's process-unique id (so a context made after a device
// reset, or a second context on the same device, gets its own lookup).  In
// host code the symbol's name is only a host-side handle, never a device
// pointer.
int32_t scratch_address(uint8_t** out) {
  static std::mutex mu;
  struct Entry {
    unsigned long long ctx_id;
    uint8_t* addr;
  };
  static Entry cache[kMaxContexts] = {};
  static int used = 0;
  unsigned long long id = 0;
  int32_t rc = current_context_id(&id);
  if (rc != MOE_OK) return rc;
  std::lock_guard<std::mutex> lock(mu);
  if (id != 0)
    for (int i = 0; i < used; ++i)
      if (cache[i].ctx_id == id) {
        *out = cache[i].addr;
        return MOE_OK;
      }
  // first call in this context (the lookup also makes the device's primary
  // context current if the thread has none yet)
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
  if (e != cudaSuccess || !p)
    return noalloc_fail(MOE_ERR_CUDA, "cudaGetSymbolAddress(g_route_scratch) failed: %s",
                        cudaGetErrorString(e));
  if (id == 0 && (rc = current_context_id(&id)) != MOE_OK) return rc;
  if (id != 0) {
    const int slot = used < kMaxContexts ? used++ : static_cast<int>(id % kMaxContexts);
    cache[slot] = Entry{id, static_cast<uint8_t*>(p)};
  }
  *out = static_cast<uint8_t*>(p);
  return MOE_OK;
}

}  // namespace

extern "C" int32_t moe_route_noalloc(const moe_shape* shape, const float* router_logits,
                                     int32_t* ids, float* weights, int32_t* offsets,
                                     int32_t* row_of, void* stream) {
  if (!shape) return noalloc_fail(MOE_ERR_INVALID_ARG, "shape is NULL");
  const int64_t T = shape->num_tokens, E = shape->num_experts, k = shape->top_k;
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 32)
    return noalloc_fail(MOE_ERR_INVALID_ARG, "need num_tokens >= 0, 1 <= num_experts <= 1024, "
                                             "1 <= top_k <= min(num_experts, 32)");
  if (T * k >= (int64_t(1) << 31))
    return noalloc_fail(MOE_ERR_INVALID_ARG, "num_tokens * top_k must be < 2^31");
  const Carve c = carve(T, E, k);
  if (c.total > MOE_NOALLOC_SCRATCH_BYTES)
    return noalloc_fail(MOE_ERR_WORKSPACE_TOO_SMALL,
                        "shape needs %zu bytes of scratch; the static scratch holds %u bytes "
                        "(use moe_forward with a caller workspace for larger shapes)",
                        c.total, static_cast<unsigned>(MOE_NOALLOC_SCRATCH_BYTES));
  if (T == 0) return MOE_OK;
  if (!router_logits || !ids || !weights || !offsets || !row_of)
    return noalloc_fail(MOE_ERR_INVALID_ARG, "a required pointer is NULL");
  const void* ptrs[5] = {router_logits, ids, weights, offsets, row_of};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) % 4 != 0)
      return noalloc_fail(MOE_ERR_MISALIGNED, "logits and outputs must be 4-byte aligned");
  // the same device check as moe_forward: sm_103a only, a clear error otherwise
  int32_t rc = moe::check_device(nullptr);
  if (rc != MOE_OK) return rc;
  uint8_t* base = nullptr;
  if ((rc = scratch_address(&base)) != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* chunk = reinterpret_cast<int32_t*>(base + c.chunk_counts);
  // Every scratch word read below is written earlier in the same call (the
  // route kernel writes the whole histogram, the scan kernel every count,
  // base and tile), so nothing needs clearing between calls.
  cudaError_t e = moe::launch_route(router_logits, static_cast<int>(T), static_cast<int>(E),
                                    static_cast<int>(k), ids, weights, chunk, nullptr, nullptr, 0,
                                    s);
  if (e == cudaSuccess)
    e = moe::launch_scan(chunk, static_cast<int>((T + moe::kRouteChunk - 1) / moe::kRouteChunk),
                         static_cast<int>(E), moe::kDecodeBN,
                         reinterpret_cast<int32_t*>(base + c.counts), offsets, chunk,
                         reinterpret_cast<int4*>(base + c.tiles),
                         reinterpret_cast<int32_t*>(base + c.num_tiles), nullptr, nullptr, s);
  if (e == cudaSuccess)
    e = moe::launch_rank(ids, chunk, static_cast<int>(T), static_cast<int>(E),
                         static_cast<int>(k), row_of,
                         reinterpret_cast<int32_t*>(base + c.token_slot), s);
  if (e != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return MOE_OK;
}
