// route.cu -- routing, expert histogram/scan + GEMM work map, and the
// expert-major scatter with fused per-token FP8 quantisation.
//
// Pages cited (title and section):
//   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
//           MXFP4xFP8 CUTLASS MoE backend for SM90": Description ("runtime
//           activation expansion and per-token FP8 quantization"; "precompute
//           grouped GEMM work scheduling ... before the main GEMM kernel"),
//           Implementation Notes (per-token activation scales computed while
//           expanding routed MoE rows; precomputed work map so the GEMM hot
//           path does no grouped tile lookup), review comments (64-bit linear
//           work index; zero routed tokens is a no-op).
//
// Kernel chain: route (one warp per token; per-chunk expert histogram) ->
// scan (one CTA: counts, offsets, per-chunk bases, GEMM tile list) ->
// quant_scatter (one CTA per token: the stable expert-major rows of its k
// slots, and its FP8 codes written to each of them).  Nothing returns to
// the host.  rank (one warp per chunk: the rows of every (token, slot)) is
// the routing-only front end's last kernel (moe_route_noalloc).
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cfloat>
#include <climits>

#include "moe_internal.h"
#include "mxfp8.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

// ---------------------------------------------------------------- routing
// Order-preserving map of a float (not NaN) to an unsigned key: a < b as
// floats exactly when key(a) < key(b) as integers; key(-inf) = 0x007FFFFF.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_order_key(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Routing of one token by one warp.  Lane l holds the logits of experts l,
// l + 32, ... (NV per lane).  k rounds of a warp argmax pick the experts in
// descending logit order, equal logits resolved toward the lower expert
// index: each round every lane offers its largest remaining logit (its
// lowest expert index among equal ones), one warp max-reduction over the
// order-preserving keys finds the round's logit and one min-reduction the
// lowest expert index offering it.  The weights are the softmax over the k
// selected logits (renormalised top-k softmax).  A NaN logit is read as
// -inf, so every round finds an expert index below E whatever the row holds.
// Lane j < k returns the j-th expert in *id and its weight in *w.
template <int NV>
__device__ __forceinline__ void route_token_warp(const float* __restrict__ row, int E, int k,
                                                 int lane, int* id, float* w) {
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -FLT_MAX;
    if (v[i] != v[i]) v[i] = -INFINITY;   // NaN ranks with -inf: k experts are always found
  }
  uint32_t taken = 0;
  float my_v = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float best = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > best || (v[i] == best && e < bi))) {
        best = v[i];
        bi = e;
      }
    }
    // a lane with nothing left to offer takes no part (key 0 is below -inf)
    const uint32_t key = bi != INT_MAX ? order_key(best) : 0u;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const uint32_t win = __reduce_min_sync(
        0xffffffffu, key == kmax ? static_cast<uint32_t>(bi) : 0xFFFFFFFFu);
    if (static_cast<int>(win & 31u) == lane) taken |= 1u << (win >> 5);
    if (lane == j) {
      my_v = from_order_key(kmax);
      my_id = static_cast<int>(win);
    }
  }
  const float lmax = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - lmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  *id = my_id;
  *w = ex / sum;
}

// One warp per token (32 warps = one chunk per CTA): route_token_warp, then
// the chunk's per-expert histogram.  The logits are the forward's input,
// complete before the previous kernel on the stream passed its own grid
// wait (every kernel here signals its dependents only after that wait), so
// the routing and the shared-memory histogram run before this kernel's
// wait, overlapping the previous forward's last kernel; every global write
// (which that kernel's reads of the workspace may still precede) follows
// the wait.
template <int NV>
__global__ void __launch_bounds__(1024) route_kernel(const float* __restrict__ logits, int T,
                                                    int E, int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts,
                                                    int32_t* __restrict__ chunk_counts,
                                                    int32_t* __restrict__ status,
                                                    int32_t* __restrict__ zero, int64_t nzero) {
  static_assert(kRouteChunk == 32, "one warp per token of the chunk");
  extern __shared__ int32_t hist[];
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteChunk + warp;
  int my_id = 0;
  float my_w = 0.f;
  if (warp < kRouteChunk && t < T) {
    route_token_warp<NV>(logits + static_cast<size_t>(t) * E, E, k, lane, &my_id, &my_w);
    if (lane < k) atomicAdd(&hist[my_id], 1);
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  // the forward's first kernel clears the device status word
  if (status && blockIdx.x == 0 && threadIdx.x == 0) {
    status[0] = 0;
    if (kChecks) {   // the work-map limits checked builds validate against
      status[2] = T * k;
      status[3] = E;
    }
  }
  if (warp < kRouteChunk && t < T && lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = my_id;
    wts[static_cast<size_t>(t) * k + lane] = my_w;
  }
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nzero;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    zero[i] = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    chunk_counts[static_cast<size_t>(blockIdx.x) * E + i] = hist[i];
}

// Exclusive scan of a pair of non-negative ints per thread over a block of up
// to 1024 threads, as one 64-bit scan of (b << 32) | a: each half's sum
// stays below 2^31, so no carry crosses between them.  Returns the
// exclusive prefixes (a, b); *total gets the block's sums.
__device__ int2 block_exclusive_scan2(int a, int b, int2* total) {
  __shared__ unsigned long long warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long v =
      (static_cast<unsigned long long>(static_cast<uint32_t>(b)) << 32) | static_cast<uint32_t>(a);
  unsigned long long x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    unsigned long long sw = lane < nw ? warp_sums[lane] : 0ull;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, sw, off);
      if (lane >= off) sw += y;
    }
    warp_sums[lane] = sw;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const unsigned long long base = warp > 0 ? warp_sums[warp - 1] : 0ull;
  const unsigned long long tot = warp_sums[((blockDim.x + 31) >> 5) - 1];
  __syncthreads();
  const unsigned long long ex = base + x - v;
  *total = make_int2(static_cast<int>(tot & 0xFFFFFFFFull), static_cast<int>(tot >> 32));
  return make_int2(static_cast<int>(ex & 0xFFFFFFFFull), static_cast<int>(ex >> 32));
}

// Row offsets and tile plan of the experts (thread e of a block with
// blockDim >= E; every thread of the block must call it; c = expert e's
// rows, 0 for e >= E).  A tile is a run of at most `bn` consecutive rows of
// one expert, as many and as large as expert_tile_plan gives for its c
// rows; one block scan of (rows, tiles) places the experts' rows and tiles
// in expert order.  With `write` the block also stores the tile list, the
// tile count and (if tile_plan is not null) the per-expert plan.
struct ExpertPlan {
  int off;          // expert e's first expanded row
  int total_rows;   // rows of all experts
  int toff;         // expert e's first tile
  int tsz;          // rows per tile
  int nt;           // tiles of expert e
  int total_tiles;  // tiles of all experts
};

__device__ ExpertPlan plan_experts(int e, int E, int c, int bn, bool write,
                                   int4* __restrict__ tiles, int32_t* __restrict__ num_tiles,
                                   int2* __restrict__ tile_plan) {
  const int2 plan = expert_tile_plan(e < E ? c : 0, bn);
  const int nt = plan.x, tsz = plan.y;
  int2 tot;
  const int2 ex = block_exclusive_scan2(e < E ? c : 0, nt, &tot);
  if (write) {
    for (int i = 0; i < nt; ++i) {
      const int r0 = i * tsz;
      tiles[ex.y + i] = make_int4(e, ex.x + r0, min(tsz, c - r0), 0);
    }
    if (tile_plan && e < E) tile_plan[e] = make_int2(ex.y, tsz);
    if (threadIdx.x == 0) *num_tiles = tot.y;
  }
  return ExpertPlan{ex.x, tot.x, ex.y, tsz, nt, tot.y};
}

// Shared memory the scan stages chunk counts in (whole chunks of E counts).
constexpr int kScanSmemBytes = 192 * 1024;

// Chunks the scan stages at a time: a multiple of 4, so that every batch
// starts on a 16-byte boundary of the count matrix.
__host__ __device__ inline int scan_batch_chunks(int E) {
  return (kScanSmemBytes / (4 * E)) & ~3;
}

// One CTA of P groups of Ep = roundup32(E) threads (P = blockDim / Ep >= 1):
// per-expert counts, offsets, per-chunk bases (stable ranks start there),
// and the GEMM tile list.  Group g sums, for its expert, the chunk counts of
// its share of the chunks; the groups' partial sums give each expert's total
// and each group's starting row.  A tile is a run of at most `bn`
// consecutive rows of one expert; an expert with c rows gets ceil(c / tsz)
// tiles of tsz = roundup16(ceil(c / ceil(c / bn))) rows, so its tiles are
// balanced and every MMA-N is a multiple of 16.
// The count matrix [num_chunks, E] comes into shared memory by bulk copies
// of up to kScanSmemBytes (one round trip per batch instead of one per
// count a thread reads); with a single batch the second pass reuses it.
// chunk_counts and chunk_base may be the same buffer (the forward turns the
// histogram into the bases in place): every count is read before the bases
// of its chunk are written, so neither pointer is declared __restrict__.
// The copy wait is bounded (status, when not null, records a timeout).
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* chunk_counts,
                                                    int num_chunks, int E, int bn,
                                                    int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets,
                                                    int32_t* chunk_base,
                                                    int4* __restrict__ tiles,
                                                    int32_t* __restrict__ num_tiles,
                                                    int2* __restrict__ tile_plan,
                                                    int32_t* __restrict__ status) {
  extern __shared__ __align__(16) int32_t staged[];   // [chunks of a batch, E]
  __shared__ int32_t part[1024];   // group g's sum for expert e at g * Ep + e
  __shared__ int32_t eoffs[1024];  // expert offsets, for every group
  __shared__ __align__(8) uint64_t bar;
  griddep_wait();
  griddep_launch_dependents();
  const int Ep = (E + 31) & ~31, P = static_cast<int>(blockDim.x) / Ep;
  const int g = static_cast<int>(threadIdx.x) / Ep, e = static_cast<int>(threadIdx.x) % Ep;
  const bool active = g < P && e < E;
  const int ch0 = active ? g * num_chunks / P : 0, ch1 = active ? (g + 1) * num_chunks / P : 0;
  const int sb = scan_batch_chunks(E), nb = (num_chunks + sb - 1) / sb;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  // batch b of chunks into shared memory (every thread calls it)
  auto stage_batch = [&](int b) {
    fence_proxy_async_smem();   // earlier reads of the buffer before the copy's writes
    __syncthreads();
    const int c0 = b * sb, nc = min(sb, num_chunks - c0);
    if (threadIdx.x == 0) {
      // whole 16-byte units: a few bytes past the matrix stay inside its
      // 256-byte-padded region
      const uint32_t bytes = (static_cast<uint32_t>(nc) * E * 4u + 15u) & ~15u;
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_load(staged, chunk_counts + static_cast<size_t>(c0) * E, bytes, &bar);
    }
    const uint32_t a = smem_u32(&bar);
    if (!mbar_try_wait(a, phase)) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait_suspend(a, phase, kSuspendNs))
        if (globaltimer_ns() - t0 > 1000000000ull) {
          if (status) atomicCAS(status, 0, kDevTimeout);
          break;
        }
    }
    phase ^= 1u;
  };
  int c = 0;
  for (int b = 0; b < nb; ++b) {
    stage_batch(b);
    const int c0 = b * sb, c1 = min(num_chunks, c0 + sb);
    for (int ch = max(ch0, c0); ch < min(ch1, c1); ++ch) c += staged[(ch - c0) * E + e];
  }
  part[threadIdx.x] = c;
  __syncthreads();
  int total = 0, gstart = 0;
  if (active)
    for (int h = 0; h < P; ++h) {
      const int v = part[h * Ep + e];
      if (h < g) gstart += v;
      total += v;
    }
  // expert offsets and the tile plan: the first group's threads are the
  // experts in order (the other groups plan nothing: "expert" E, 0 rows)
  const ExpertPlan pl = plan_experts(g == 0 ? e : E, E, g == 0 && e < E ? total : 0, bn, true,
                                     tiles, num_tiles, tile_plan);
  const int off = pl.off;
  if (g == 0) eoffs[e] = off;
  __syncthreads();
  if (g == 0 && e < E) {
    counts[e] = total;
    offsets[e] = off;
  }
  if (threadIdx.x == 0) offsets[E] = pl.total_rows;
  int run = active ? eoffs[e] + gstart : 0;
  for (int b = 0; b < nb; ++b) {
    if (nb > 1) stage_batch(b);   // a single batch is still staged
    const int c0 = b * sb, c1 = min(num_chunks, c0 + sb);
    for (int ch = max(ch0, c0); ch < min(ch1, c1); ++ch) {
      const int cc = staged[(ch - c0) * E + e];
      chunk_base[static_cast<size_t>(ch) * E + e] = run;
      run += cc;
    }
  }
}

// One warp per chunk of kRouteChunk tokens: the warp stages the chunk's
// routed experts and per-expert bases in shared memory, then walks the
// chunk's tokens in order and hands out rows from the bases (a token's k
// experts are distinct, so the k lanes never collide), which makes each
// expert's rows ascend in token order.
__global__ void __launch_bounds__(256) rank_kernel(const int32_t* __restrict__ ids,
                                                   const int32_t* __restrict__ chunk_base,
                                                   int T, int E, int k, int num_chunks,
                                                   int32_t* __restrict__ row_of,
                                                   int32_t* __restrict__ token_slot) {
  extern __shared__ int32_t sm[];
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * (blockDim.x >> 5) + warp;
  if (chunk >= num_chunks) return;
  int32_t* base = sm + warp * (E + kRouteChunk * k);
  int32_t* cid = base + E;
  const int t0 = chunk * kRouteChunk, nt = min(kRouteChunk, T - t0);
  for (int i = lane; i < E; i += 32) base[i] = chunk_base[static_cast<size_t>(chunk) * E + i];
  for (int i = lane; i < nt * k; i += 32) cid[i] = ids[static_cast<size_t>(t0) * k + i];
  __syncwarp();
  for (int tt = 0; tt < nt; ++tt) {
    if (lane < k) {
      const size_t ts = static_cast<size_t>(t0 + tt) * k + lane;
      const int e = cid[tt * k + lane];
      const int r = base[e];
      base[e] = r + 1;
      row_of[ts] = r;
      token_slot[r] = static_cast<int32_t>(ts);
    }
    __syncwarp();
  }
}

// Quantises token t's row of x (H bf16) with the block's threads and writes
// the codes to the k expanded rows rows[0..k): amax -> s = amax/448, inv =
// 448/amax (IEEE divisions) -> E4M3 codes of x*inv (round to nearest even,
// satfinite); an all-zero row gets s = 1 and zero codes.  `warp_max` holds
// one float per warp of the block.  A thread keeps its first KEEP 16-element
// vectors in registers between the amax pass and the conversion (the row is
// read once when H <= 16 * KEEP * blockDim).

__device__ __forceinline__ uint4 fp8_codes16(const uint4 (&q)[2], float inv) {
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
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int KEEP>
__device__ void quantize_token(const __nv_bfloat16* __restrict__ x, int t, int k, int H,
                               const int32_t* rows, float* warp_max, uint8_t* __restrict__ xq,
                               float* __restrict__ x_scale) {
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
  const int nvec = H / 16;  // 16 elements (two 16-byte loads) per thread step
  uint4 keep[KEEP][2];
  float amax = 0.f;
  int it = 0;
  for (int i = threadIdx.x; i < nvec; i += blockDim.x, ++it) {
    uint4 q[2] = {__ldg(xr + 2 * i), __ldg(xr + 2 * i + 1)};
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(q);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
#pragma unroll
    for (int c = 0; c < KEEP; ++c)
      if (c == it) {
        keep[c][0] = q[0];
        keep[c][1] = q[1];
      }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) amax = fmaxf(amax, warp_max[w]);
  const bool nz = amax > 0.f;
  const float s = nz ? amax / 448.0f : 1.0f;
  const float inv = nz ? 448.0f / amax : 0.0f;
  it = 0;
  for (int i = threadIdx.x; i < nvec; i += blockDim.x, ++it) {
    uint4 out = make_uint4(0, 0, 0, 0);
    if (nz) {
      uint4 q[2];
      if (it < KEEP) {
#pragma unroll
        for (int c = 0; c < KEEP; ++c)
          if (c == it) {
            q[0] = keep[c][0];
            q[1] = keep[c][1];
          }
      } else {
        q[0] = __ldg(xr + 2 * i);
        q[1] = __ldg(xr + 2 * i + 1);
      }
      out = fp8_codes16(q, inv);
    }
    for (int j = 0; j < k; ++j)
      reinterpret_cast<uint4*>(xq + static_cast<size_t>(rows[j]) * H)[i] = out;
  }
  if (static_cast<int>(threadIdx.x) < k) x_scale[rows[threadIdx.x]] = s;
}

// quantize_token on a row already staged in shared memory (xs: H bf16): the
// same arithmetic, both passes reading shared memory.  code_row >= 0: the
// codes go to that one row of xq only (the token-major copy GEMM1 gathers
// from); the scale still goes to the k rows.
__device__ void quantize_token_staged(const __nv_bfloat16* xs, int k, int H, const int32_t* rows,
                                      float* warp_max, uint8_t* __restrict__ xq,
                                      float* __restrict__ x_scale, int code_row = -1) {
  const uint4* xr = reinterpret_cast<const uint4*>(xs);
  const int nvec = H / 16;
  float amax = 0.f;
  for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
    const uint4 q[2] = {xr[2 * i], xr[2 * i + 1]};
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(q);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) amax = fmaxf(amax, warp_max[w]);
  const bool nz = amax > 0.f;
  const float s = nz ? amax / 448.0f : 1.0f;
  const float inv = nz ? 448.0f / amax : 0.0f;
  for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
    uint4 out = make_uint4(0, 0, 0, 0);
    if (nz) {
      const uint4 q[2] = {xr[2 * i], xr[2 * i + 1]};
      out = fp8_codes16(q, inv);
    }
    if (code_row >= 0)
      reinterpret_cast<uint4*>(xq + static_cast<size_t>(code_row) * H)[i] = out;
    else
      for (int j = 0; j < k; ++j)
        reinterpret_cast<uint4*>(xq + static_cast<size_t>(rows[j]) * H)[i] = out;
  }
  if (static_cast<int>(threadIdx.x) < k) x_scale[rows[threadIdx.x]] = s;
}

// MXFP8 (the W8A8 mode) quantisation of a token's row xrow (global or
// shared memory), per 32-element
// block: X = 2^clamp(floor(log2 amax) - 8, -127, 127) (8 = E4M3's emax),
// codes = E4M3_rne_satfinite(x / X), scale byte = exponent + 127; an
// all-zero block gets byte 127 (its codes are those of +-0).  Dividing by a
// power of two is exact, so x * 2^-e rounds once, in the conversion.  Codes
// go to the k expanded rows; scale bytes to the row-major x_sf [R, H/32] and
// to the GEMM's per-tile layout at sfb_base[j] + (b / 4) * kSfbTileBytes +
// b % 4 for block b of row rows[j].
// SPLIT (the W4A16 mode): the two-term split of each block (split_block),
// in rows of 2H codes -- hi blocks in columns [0, H), lo blocks in [H, 2H)
// -- whose scale bytes follow the same order in x_sf [R, 2H/32] (block H/32
// + b is b's lo term); in the per-tile layout the lo byte sits kSfbLoOffset
// after the hi byte.
template <bool SPLIT>
__device__ void quantize_token_mx(const __nv_bfloat16* xrow, int k, int H, const int32_t* rows,
                                  const int64_t* sfb_base, uint8_t* __restrict__ xq,
                                  uint8_t* __restrict__ x_sf, uint8_t* __restrict__ sfb) {
  const uint4* xr = reinterpret_cast<const uint4*>(xrow);   // the token's row (global or shared)
  const int nblk = H / 32;
  const int64_t W = SPLIT ? 2 * H : H, nsf = SPLIT ? 2 * nblk : nblk;
  for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
    uint4 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = xr[4 * b + i];
    uint8_t sbyte, lbyte = 0;
    uint4 codes[2], lcodes[2];
    if constexpr (SPLIT)
      split_block(q, &sbyte, codes, &lbyte, lcodes);
    else
      mx_quant_block(q, &sbyte, codes);
    for (int j = 0; j < k; ++j) {
      const int64_t r = rows[j];
      uint4* dst = reinterpret_cast<uint4*>(xq + r * W + 32 * b);
      dst[0] = codes[0];
      dst[1] = codes[1];
      x_sf[r * nsf + b] = sbyte;
      sfb[sfb_base[j] + static_cast<int64_t>(b >> 2) * kSfbTileBytes + (b & 3)] = sbyte;
      if constexpr (SPLIT) {
        uint4* ldst = reinterpret_cast<uint4*>(xq + r * W + H + 32 * b);
        ldst[0] = lcodes[0];
        ldst[1] = lcodes[1];
        x_sf[r * nsf + nblk + b] = lbyte;
        sfb[sfb_base[j] + static_cast<int64_t>(b >> 2) * kSfbTileBytes + kSfbLoOffset + (b & 3)] =
            lbyte;
      }
    }
  }
}

// quantize_token_mx with 8 lanes per 32-element block (lane l of the warp
// holds elements 4 (l % 8) .. + 3 of block 4 w' + l / 8, w' the warp's
// iteration) instead of one thread: few registers per thread, so that two
// 1024-thread CTAs of the small-batch kernel fit an SM.  The same codes and
// scale bytes.
template <bool SPLIT>
__device__ void quantize_token_mx_lanes(const __nv_bfloat16* __restrict__ x, int t, int k, int H,
                                        const int32_t* rows, const int64_t* sfb_base,
                                        uint8_t* __restrict__ xq, uint8_t* __restrict__ x_sf,
                                        uint8_t* __restrict__ sfb) {
  const int lane = threadIdx.x & 31, sub = lane & 7;
  const int nblk = H / 32;   // a multiple of 4
  const int64_t W = SPLIT ? 2 * H : H, nsf = SPLIT ? 2 * nblk : nblk;
  for (int b = 4 * (threadIdx.x >> 5) + (lane >> 3); b < nblk; b += 4 * (blockDim.x >> 5)) {
    const int c0 = 32 * b + 4 * sub;   // the lane's first column
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(x + static_cast<size_t>(t) * H + c0));
    const float2 f01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 f23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    float v[4] = {f01.x, f01.y, f23.x, f23.y}, dec[4];
    uint8_t sbyte, lbyte = 0;
    const uint32_t c = mx_quad_term(v, SPLIT ? 7 : 8, &sbyte, dec);
    uint32_t lc = 0;
    if constexpr (SPLIT) {
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __fsub_rn(v[i], dec[i]);
      lc = mx_quad_term(v, 7, &lbyte, dec);
    }
    for (int j = 0; j < k; ++j) {
      const int64_t r = rows[j];
      const int64_t sb = sfb_base[j] + static_cast<int64_t>(b >> 2) * kSfbTileBytes + (b & 3);
      *reinterpret_cast<uint32_t*>(xq + r * W + c0) = c;
      if (sub == 0) {
        x_sf[r * nsf + b] = sbyte;
        sfb[sb] = sbyte;
      }
      if constexpr (SPLIT) {
        *reinterpret_cast<uint32_t*>(xq + r * W + H + c0) = lc;
        if (sub == 1) {
          x_sf[r * nsf + nblk + b] = lbyte;
          sfb[sb + kSfbLoOffset] = lbyte;
        }
      }
    }
  }
}

// One CTA per token t: the rows of its k slots, then the quantisation of
// the token into them (AQ: per-row FP8, MXFP8 or the two-term split).
// stage_x (x in device memory): the token's row comes into shared memory by
// one bulk copy issued before the grid dependency wait --
// x is the forward's input, complete before the forward's first kernel
// passed its own wait, hence before this grid started -- so the copy
// overlaps the wait and the ranking.  Slot j's row is the chunk's base row for its expert e (from the
// scan) plus the number of the chunk's earlier tokens routed to e -- the
// stable, ascending-token order inside each expert (a token's k experts are
// distinct).  The CTA writes row_of and token_slot for its slots.
template <int AQ>
__global__ void __launch_bounds__(256) quant_scatter_kernel(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ chunk_base,
    const int32_t* __restrict__ ids, const int32_t* __restrict__ offsets,
    const int2* __restrict__ tile_plan, int E, int k, int H, int32_t* __restrict__ row_of,
    int32_t* __restrict__ token_slot, uint8_t* __restrict__ xq, float* __restrict__ x_scale,
    uint8_t* __restrict__ x_sf, uint8_t* __restrict__ sfb, int stage_x,
    int32_t* __restrict__ status, int token_major) {
  extern __shared__ __align__(128) uint8_t xstage[];
  __shared__ int32_t rows[32];
  __shared__ int32_t my_e[32];
  __shared__ int32_t before[32];
  __shared__ int64_t sfb_base[32];
  __shared__ float warp_max[32];
  __shared__ __align__(8) uint64_t xbar;
  const int t = blockIdx.x;
  const bool staged = stage_x != 0;
  if (staged && threadIdx.x == 0) {
    mbar_init(&xbar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&xbar, static_cast<uint32_t>(H) * 2u);
    bulk_load(xstage, x + static_cast<size_t>(t) * H, static_cast<uint32_t>(H) * 2u, &xbar);
  }
  griddep_wait();
  griddep_launch_dependents();
  const int chunk = t / kRouteChunk, t0 = chunk * kRouteChunk;
  if (static_cast<int>(threadIdx.x) < k) {
    my_e[threadIdx.x] = ids[static_cast<size_t>(t) * k + threadIdx.x];
    before[threadIdx.x] = 0;
  }
  __syncthreads();
  // the chunk's earlier (token, slot) entries routed to each of t's experts
  for (int i = threadIdx.x; i < (t - t0) * k; i += blockDim.x) {
    const int ei = ids[static_cast<size_t>(t0) * k + i];
    for (int j = 0; j < k; ++j)
      if (my_e[j] == ei) atomicAdd(&before[j], 1);
  }
  __syncthreads();
  if (static_cast<int>(threadIdx.x) < k) {
    const int j = threadIdx.x;
    const size_t ts = static_cast<size_t>(t) * k + j;
    const int e = my_e[j];
    const int r = chunk_base[static_cast<size_t>(chunk) * E + e] + before[j];
    rows[j] = r;
    row_of[ts] = r;
    token_slot[r] = static_cast<int32_t>(ts);
    if (AQ != kActFp8Row)
      sfb_base[j] = sfb_row_base(r, offsets[e], tile_plan[e], H / kTileK);
  }
  __syncthreads();
  const __nv_bfloat16* xs = reinterpret_cast<const __nv_bfloat16*>(xstage);
  if (staged) {
    int32_t none = 0;
    if (!mbar_wait(&xbar, 0, 1000000000ull, status, kDevTimeout, &none)) return;
  }
  if constexpr (AQ == kActFp8Row) {
    if (staged)
      quantize_token_staged(xs, k, H, rows, warp_max, xq, x_scale, token_major ? t : -1);
    else
      quantize_token<2>(x, t, k, H, rows, warp_max, xq, x_scale);   // 256 threads
  } else {
    quantize_token_mx<AQ == kActSplit>(staged ? xs : x + static_cast<size_t>(t) * H, k, H, rows,
                                       sfb_base, xq, x_sf, sfb);
  }
}

// Small batches (T <= kSmallT = 256): one kernel replaces scan +
// quant_scatter.  CTA t (1024 threads, one expert per thread) rebuilds the
// per-expert counts and offsets from all T*k routed ids in shared memory,
// ranks its own token's k slots (rank of (t, e) = number of earlier tokens
// routed to e, i.e. stable ascending token order), writes their rows, and
// quantises its token into them.  CTA 0 also writes counts, offsets and the
// GEMM tile list.  The redundant O(T*k) counting per CTA is cheap at these
// sizes and removes three launches from the decode path.
template <int AQ>
__global__ void __launch_bounds__(1024, 2) expand_small_kernel(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ ids, int T, int E, int k,
    int H, int bn, int32_t* __restrict__ counts_out, int32_t* __restrict__ offsets_out,
    int4* __restrict__ tiles, int32_t* __restrict__ num_tiles, int2* __restrict__ tile_plan,
    int32_t* __restrict__ row_of, int32_t* __restrict__ token_slot, uint8_t* __restrict__ xq,
    float* __restrict__ x_scale, uint8_t* __restrict__ x_sf, uint8_t* __restrict__ sfb) {
  extern __shared__ int32_t sm[];
  int2* plan = reinterpret_cast<int2*>(sm);   // [E] tile plan (MXFP8)
  int32_t* cnt = sm + 2 * E;    // [E]
  int32_t* my_e = cnt + E;      // [k] experts of this token
  int32_t* my_rank = my_e + 32; // [k]
  int32_t* rows = my_rank + 32; // [k]
  __shared__ float warp_max[32];
  __shared__ int64_t sfb_base[32];
  griddep_wait();
  griddep_launch_dependents();
  const int t = blockIdx.x, e = threadIdx.x;
  if (e < E) cnt[e] = 0;
  if (e < k) {
    my_e[e] = ids[static_cast<size_t>(t) * k + e];
    my_rank[e] = 0;
  }
  __syncthreads();
  const int n = T * k, mine = t * k;   // ids of earlier tokens are [0, mine)
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int ei = ids[i];
    atomicAdd(&cnt[ei], 1);
    if (i < mine)
      for (int j = 0; j < k; ++j)
        if (my_e[j] == ei) atomicAdd(&my_rank[j], 1);
  }
  __syncthreads();
  const int c = e < E ? cnt[e] : 0;
  // every CTA plans the rows and tiles (its rows' positions); CTA 0 writes
  // the tile list
  const ExpertPlan pl = plan_experts(e, E, c, bn, t == 0, tiles, num_tiles, tile_plan);
  const int off = pl.off, total_rows = pl.total_rows;
  if (e < E) cnt[e] = off;     // cnt now holds the offsets
  if (AQ != kActFp8Row && e < E) plan[e] = make_int2(pl.toff, pl.tsz);
  __syncthreads();
  if (e < k) {
    const size_t ts = static_cast<size_t>(t) * k + e;
    const int r = cnt[my_e[e]] + my_rank[e];
    rows[e] = r;
    row_of[ts] = r;
    token_slot[r] = static_cast<int32_t>(ts);
  }
  if (t == 0) {
    if (e < E) {
      counts_out[e] = c;
      offsets_out[e] = off;
    }
    if (e == 0) offsets_out[E] = total_rows;
  }
  __syncthreads();
  if constexpr (AQ == kActFp8Row) {
    quantize_token<1>(x, t, k, H, rows, warp_max, xq, x_scale);   // 1024 threads
  } else {
    if (e < k)
      sfb_base[e] = sfb_row_base(rows[e], cnt[my_e[e]], plan[my_e[e]], H / kTileK);
    __syncthreads();
    quantize_token_mx_lanes<AQ == kActSplit>(x, t, k, H, rows, sfb_base, xq, x_sf, sfb);
  }
}

// Tiny batches (T <= kTinyT, W4A8): routing, expansion and quantisation in
// one kernel of T CTAs (1024 threads each), so the routed rows need no
// second launch and each token row is fetched while the routing runs.
// CTA t:
//   1. prefetches token t's row into L2; warp w routes token w (every CTA
//      routes all T tokens -- the same selection and softmax as
//      route_kernel; the logits are L2-resident after the first CTA) and
//      counts its experts (shared atomics) -- all before the grid wait, as
//      in route_kernel: logits and x are the forward's inputs;
//   2. after the wait: offsets (block scan), the tile plan and the stable
//      rank of token t's slots (earlier tokens routed to the same expert);
//      CTA 0 writes counts, offsets and the tile list;
//   3. quantises token t into its k rows (quantize_token).
template <int NV>
__global__ void __launch_bounds__(1024) route_expand_tiny_kernel(
    const float* __restrict__ logits, const __nv_bfloat16* __restrict__ x, int T, int E, int k,
    int H, int bn, int32_t* __restrict__ ids, float* __restrict__ wts,
    int32_t* __restrict__ counts_out, int32_t* __restrict__ offsets_out, int4* __restrict__ tiles,
    int32_t* __restrict__ num_tiles, int2* __restrict__ tile_plan, int32_t* __restrict__ row_of,
    int32_t* __restrict__ token_slot, uint8_t* __restrict__ xq, float* __restrict__ x_scale,
    int32_t* __restrict__ status, const TinyPrefetch pf, int32_t* __restrict__ zero,
    int64_t nzero) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                        // [E] counts, then offsets
  int32_t* sid = sm + E;                    // [kTinyT * 32] routed experts
  __shared__ int32_t rows[32];
  __shared__ float warp_max[32];
  __shared__ int32_t tile_expert[kTinyPrefetchTiles];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (t >= T) {
    // ---------------------------------------------------- prefetch CTAs
    // Route the T tokens like the CTAs below, plan the tiles without
    // writing them, and ask L2 for the first weight boxes (and their scale
    // blocks) of the GEMM1 items that run first: items 0 .. first_items-1,
    // item i = tile i / MT, M-tile i % MT.  Only inputs are read and
    // nothing is written, so these CTAs never wait for the previous grid:
    // the weight stream starts while the front end (and the previous
    // forward's last kernel) runs.
    for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    if (warp < T) {
      int my_id;
      float my_w;
      route_token_warp<NV>(logits + static_cast<size_t>(warp) * E, E, k, lane, &my_id, &my_w);
      if (lane < k) atomicAdd(&cnt[my_id], 1);
    }
    __syncthreads();
    const int e = threadIdx.x;
    const ExpertPlan pl = plan_experts(e, E, e < E ? cnt[e] : 0, bn, false, nullptr, nullptr,
                                       nullptr);
    if (e < E)
      for (int i = 0; i < pl.nt && pl.toff + i < kTinyPrefetchTiles; ++i)
        tile_expert[pl.toff + i] = e;
    __syncthreads();
    const int ntiles = min(pl.total_tiles, kTinyPrefetchTiles);
    const int items = min(pf.first_items, ntiles * pf.mt);
    const int nb = min(pf.boxes, pf.ks);
    const int p = t - T, np = static_cast<int>(gridDim.x) - T;
    for (int idx = threadIdx.x; idx < items * nb; idx += blockDim.x) {
      const int it = p + (idx / nb) * np;   // this CTA's items: p, p + np, ...
      if (it >= items) continue;
      const int ks = idx % nb;
      const int64_t box =
          (static_cast<int64_t>(tile_expert[it / pf.mt]) * pf.mt + it % pf.mt) * pf.ks + ks;
      bulk_prefetch_l2(pf.w + box * kFp4BoxBytes, kFp4BoxBytes);
      bulk_prefetch_l2(pf.sf + box * 512, 512u);
    }
    return;
  }
  {   // L2 prefetch of token t's row (2H bytes), 128-byte lines
    const char* base = reinterpret_cast<const char*>(x + static_cast<size_t>(t) * H);
    for (int i = threadIdx.x; i < (2 * H + 127) / 128; i += blockDim.x)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(base + static_cast<size_t>(i) * 128));
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  int my_id = 0;
  float my_w = 0.f;
  if (warp < T) {
    route_token_warp<NV>(logits + static_cast<size_t>(warp) * E, E, k, lane, &my_id, &my_w);
    if (lane < k) {
      sid[warp * 32 + lane] = my_id;
      atomicAdd(&cnt[my_id], 1);
    }
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  if (t == 0 && threadIdx.x == 0) {   // first kernel of the forward
    status[0] = 0;
    if (kChecks) {
      status[2] = T * k;
      status[3] = E;
    }
  }
  if (warp == t && lane < k) {
    const size_t ts = static_cast<size_t>(warp) * k + lane;
    ids[ts] = my_id;
    wts[ts] = my_w;
  }
  for (int64_t i = static_cast<int64_t>(t) * blockDim.x + threadIdx.x; i < nzero;
       i += static_cast<int64_t>(T) * blockDim.x)
    zero[i] = 0;
  // counts -> offsets and the tile list (one block scan)
  const int e = threadIdx.x;
  const int c = e < E ? cnt[e] : 0;
  const ExpertPlan pl = plan_experts(e, E, c, bn, t == 0, tiles, num_tiles, tile_plan);
  if (e < E) cnt[e] = pl.off;
  if (t == 0) {
    if (e < E) {
      counts_out[e] = c;
      offsets_out[e] = pl.off;
    }
    if (e == 0) offsets_out[E] = pl.total_rows;
  }
  __syncthreads();
  // token t's rows: stable rank among earlier tokens routed to the same expert
  if (threadIdx.x < k) {
    const int j = threadIdx.x;
    const int ej = sid[t * 32 + j];
    int rank = 0;
    for (int t2 = 0; t2 < t; ++t2)
      for (int j2 = 0; j2 < k; ++j2) rank += sid[t2 * 32 + j2] == ej;
    const int r = cnt[ej] + rank;
    rows[j] = r;
    row_of[static_cast<size_t>(t) * k + j] = r;
    token_slot[r] = t * k + j;
  }
  __syncthreads();
  quantize_token<1>(x, t, k, H, rows, warp_max, xq, x_scale);   // 1024 threads
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* wts,
                         int32_t* chunk_counts, int32_t* status, int32_t* zero, int64_t nzero,
                         cudaStream_t s) {
  const int chunks = (T + kRouteChunk - 1) / kRouteChunk;
  const size_t smem = static_cast<size_t>(E) * sizeof(int32_t);
  const int nv = (E + 31) / 32;
  auto kern = nv <= 1 ? route_kernel<1> : nv <= 2 ? route_kernel<2> : nv <= 4 ? route_kernel<4>
            : nv <= 8 ? route_kernel<8> : nv <= 16 ? route_kernel<16> : route_kernel<32>;
  return launch_pdl(kern, dim3(chunks), dim3(1024), smem, s, logits, T, E, k, ids, wts,
                    chunk_counts, status, zero, zero ? nzero : int64_t{0});
}

cudaError_t launch_route_expand_tiny(const float* logits, const void* x, int T, int E, int k,
                                     int H, int bn, int32_t* ids, float* wts, int32_t* counts,
                                     int32_t* offsets, int4* tiles, int32_t* num_tiles,
                                     int2* tile_plan, int32_t* row_of, int32_t* token_slot,
                                     uint8_t* xq, float* x_scale, int32_t* status,
                                     const TinyPrefetch& pf, int32_t* zero, int64_t nzero,
                                     cudaStream_t s) {
  const size_t smem = static_cast<size_t>(E + kTinyT * 32) * sizeof(int32_t);
  const int nv = (E + 31) / 32;
  auto kern = nv <= 1 ? route_expand_tiny_kernel<1> : nv <= 2 ? route_expand_tiny_kernel<2>
            : nv <= 4 ? route_expand_tiny_kernel<4> : nv <= 8 ? route_expand_tiny_kernel<8>
            : nv <= 16 ? route_expand_tiny_kernel<16> : route_expand_tiny_kernel<32>;
  const bool on = pf.w && pf.sf && pf.ctas > 0 && pf.boxes > 0 && pf.first_items > 0 &&
                  pf.mt > 0 && pf.ks > 0;
  return launch_pdl(kern, dim3(T + (on ? pf.ctas : 0)), dim3(1024), smem, s, logits,
                    static_cast<const __nv_bfloat16*>(x), T, E, k, H, bn, ids, wts, counts,
                    offsets, tiles, num_tiles, tile_plan, row_of, token_slot, xq, x_scale, status,
                    pf, zero, zero ? nzero : int64_t{0});
}

cudaError_t launch_scan(const int32_t* chunk_counts, int num_chunks, int E, int bn,
                        int32_t* counts, int32_t* offsets, int32_t* chunk_base, int4* tiles,
                        int32_t* num_tiles, int2* tile_plan, int32_t* status, cudaStream_t s) {
  const int ep = ((E + 31) / 32) * 32;    // one group of threads per expert set
  const int threads = (1024 / ep) * ep;   // as many groups as fit 1024 threads
  static DeviceOnce smem_set;
  cudaError_t e = set_smem_limit_once(scan_kernel, kScanSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const int sb = scan_batch_chunks(E);
  const size_t smem =
      (static_cast<size_t>(std::min(num_chunks, sb)) * E * 4 + 15) / 16 * 16;
  return launch_pdl(scan_kernel, dim3(1), dim3(threads), smem, s, chunk_counts, num_chunks, E,
                    bn, counts, offsets, chunk_base, tiles, num_tiles, tile_plan, status);
}

cudaError_t launch_rank(const int32_t* ids, const int32_t* chunk_base, int T, int E, int k,
                        int32_t* row_of, int32_t* token_slot, cudaStream_t s) {
  const int chunks = (T + kRouteChunk - 1) / kRouteChunk;
  // per warp: the chunk's per-expert bases and its routed experts
  const size_t per_warp = static_cast<size_t>(E + kRouteChunk * k) * sizeof(int32_t);
  const int warps = static_cast<int>(std::min<size_t>(8, 49152 / per_warp));
  const size_t smem = static_cast<size_t>(warps) * per_warp;
  return launch_pdl(rank_kernel, dim3((chunks + warps - 1) / warps), dim3(32 * warps), smem, s,
                    ids, chunk_base, T, E, k, chunks, row_of, token_slot);
}

cudaError_t launch_quant_scatter(const void* x, bool x_on_device, const int32_t* chunk_base,
                                 const int32_t* ids, const int32_t* offsets, const int2* tile_plan,
                                 int T, int E, int k, int H, int32_t* row_of, int32_t* token_slot,
                                 const QuantOut& q, int32_t* status, cudaStream_t s) {
  auto kern = q.act == kActSplit    ? quant_scatter_kernel<kActSplit>
              : q.act == kActMxfp8 ? quant_scatter_kernel<kActMxfp8>
                                   : quant_scatter_kernel<kActFp8Row>;
  // the staged row within the default shared-memory limit (48 KB)
  const bool stage = x_on_device && H * 2 <= 48 * 1024;
  if (q.token_major && (!stage || q.act != kActFp8Row)) return cudaErrorInvalidValue;
  return launch_pdl(kern, dim3(T), dim3(256), stage ? static_cast<size_t>(H) * 2 : 0, s,
                    static_cast<const __nv_bfloat16*>(x), chunk_base, ids, offsets, tile_plan, E,
                    k, H, row_of, token_slot, q.xq, q.x_scale, q.x_sf, q.sfb, stage ? 1 : 0,
                    status, q.token_major ? 1 : 0);
}

cudaError_t launch_expand_small(const void* x, const int32_t* ids, int T, int E, int k, int H,
                                int bn, int32_t* counts, int32_t* offsets, int4* tiles,
                                int32_t* num_tiles, int2* tile_plan, int32_t* row_of,
                                int32_t* token_slot, const QuantOut& q, cudaStream_t s) {
  // plan int2[E], cnt[E], my_e/my_rank/rows [32] each
  const size_t smem = static_cast<size_t>(3 * E + 96) * sizeof(int32_t);
  auto kern = q.act == kActSplit    ? expand_small_kernel<kActSplit>
              : q.act == kActMxfp8 ? expand_small_kernel<kActMxfp8>
                                   : expand_small_kernel<kActFp8Row>;
  return launch_pdl(kern, dim3(T), dim3(1024), smem, s, static_cast<const __nv_bfloat16*>(x),
                    ids, T, E, k, H, bn, counts, offsets, tiles, num_tiles, tile_plan, row_of,
                    token_slot, q.xq, q.x_scale, q.x_sf, q.sfb);
}

}  // namespace moe
