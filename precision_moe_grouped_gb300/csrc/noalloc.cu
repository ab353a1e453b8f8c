// noalloc.cu -- moe_route_noalloc: the routing front end of the forward
// (top-k routing, per-expert offsets, expert-major row map) for callers that
// cannot allocate device memory.
//
// Its scratch (the per-chunk expert histogram, per-expert counts, the row ->
// (token, slot) map and the GEMM tile list the scan kernel also writes) lives
// in one file-scope device array instead of a caller workspace.  The array
// is part of the library image: every GPU that loads the library holds it
// until the process exits.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

__device__ __align__(256) uint8_t g_route_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

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

// Device address of g_route_scratch on the current device, looked up once
// per device with that device current.  In host code the symbol's name is
// only a host-side handle, never a device pointer.
int32_t scratch_address(uint8_t** out) {
  static std::mutex mu;
  static uint8_t* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(MOE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || !p)
      return noalloc_fail(MOE_ERR_CUDA, "cudaGetSymbolAddress(g_route_scratch) failed: %s",
                          cudaGetErrorString(e));
    addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = addr[dev];
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
  uint8_t* base = nullptr;
  int32_t rc = scratch_address(&base);
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* chunk = reinterpret_cast<int32_t*>(base + c.chunk_counts);
  // Every scratch word read below is written earlier in the same call (the
  // route kernel writes the whole histogram, the scan kernel every count,
  // base and tile), so nothing needs clearing between calls.
  cudaError_t e = moe::launch_route(router_logits, static_cast<int>(T), static_cast<int>(E),
                                    static_cast<int>(k), ids, weights, chunk, nullptr, s);
  if (e == cudaSuccess)
    e = moe::launch_scan(chunk, static_cast<int>((T + moe::kRouteChunk - 1) / moe::kRouteChunk),
                         static_cast<int>(E), moe::kDecodeBN,
                         reinterpret_cast<int32_t*>(base + c.counts), offsets, chunk,
                         reinterpret_cast<int4*>(base + c.tiles),
                         reinterpret_cast<int32_t*>(base + c.num_tiles), nullptr, s);
  if (e == cudaSuccess)
    e = moe::launch_rank(ids, chunk, static_cast<int>(T), static_cast<int>(E),
                         static_cast<int>(k), row_of,
                         reinterpret_cast<int32_t*>(base + c.token_slot), s);
  if (e != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return MOE_OK;
}
