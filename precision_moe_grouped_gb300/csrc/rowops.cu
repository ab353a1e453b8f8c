// rowops.cu -- the memory-bound row kernels between and after the GEMMs:
// per-row FP8 quantisation of h (GEMM2's input), the top-k weighted combine,
// and the bounded-wait self test (the h quantisation's per-row arithmetic:
// rowops.cuh).
//
// Pages cited (title and section):
//   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
//           MXFP4xFP8 CUTLASS MoE backend for SM90": Description (per-token FP8
//           scales threaded through activation and GEMM1/GEMM2), review
//           comments (FP8 x MXFP4 quant params carry fc1 and fc2 token scales).
//   [P4793] flashinfer PR #4793, "Unify MoE CuTe DSL dispatch to be dtype
//           agnostic": walkthrough (grouped GEMM with finalize fusion: the
//           top-k weighted un-permute of the expert outputs).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "moe_internal.h"
#include "mxfp8.cuh"
#include "ptx.cuh"
#include "rowops.cuh"

namespace moe {

namespace {

// One warp per expanded row of h (bf16 [R, I]): hquant_row_warp.  GEMM2
// may launch as soon as these blocks have started: it streams its weights
// while this kernel waits for GEMM1 and quantises, and waits for this
// kernel's results itself.  (The form for rows too long to stage.)
__global__ void __launch_bounds__(256) hquant_kernel(const __nv_bfloat16* __restrict__ h, int R,
                                                     int I, uint8_t* __restrict__ hq,
                                                     float* __restrict__ h_scale) {
  griddep_launch_dependents();
  griddep_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (warp >= R) return;
  hquant_row_warp(h, warp, I, hq, h_scale, threadIdx.x & 31);
}

// Rows of h one staged block holds, and the longest row staged.
constexpr int kHqStageRows = 8;
constexpr int kHqStageMaxI = 4096;   // 8 rows x 8 KB = 64 KB of shared memory

// The same quantisation with the block's kHqStageRows consecutive rows
// brought into shared memory by one bulk copy (up to 64 KB in flight per
// block, several blocks per SM), then one warp per row (hquant_row_smem).
// A timed-out wait for the copy records MOE_ERR_DEVICE_TIMEOUT in status.
__global__ void __launch_bounds__(256) hquant_staged_kernel(const __nv_bfloat16* __restrict__ h,
                                                            int R, int I,
                                                            uint8_t* __restrict__ hq,
                                                            float* __restrict__ h_scale,
                                                            int32_t* __restrict__ status,
                                                            uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t hstage[];
  __shared__ __align__(8) uint64_t bar;
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  griddep_wait();
  const int r0 = blockIdx.x * kHqStageRows;
  const int nr = min(kHqStageRows, R - r0);
  if (threadIdx.x == 0) {
    const uint32_t bytes = static_cast<uint32_t>(nr) * static_cast<uint32_t>(I) * 2u;
    mbar_arrive_expect_tx(&bar, bytes);
    bulk_load(hstage, h + static_cast<size_t>(r0) * I, bytes, &bar);
  }
  int32_t none = 0;
  if (!mbar_wait(&bar, 0, timeout_ns, status, kDevTimeout, &none)) return;
  const int warp = threadIdx.x >> 5;
  if (warp < nr)
    hquant_row_smem(reinterpret_cast<const __nv_bfloat16*>(hstage) + static_cast<size_t>(warp) * I,
                    r0 + warp, I, hq, h_scale, threadIdx.x & 31);
}

// MXFP8 (the W8A8 mode) quantisation of h, or (SPLIT, the W4A16 mode) its
// two-term split: one warp per expanded row r, lane l converts the
// 32-element blocks l, l + 32, ...; codes to hq (rows of I codes, or 2I
// with the lo terms in columns [I, 2I)), scale bytes to the row-major h_sf
// [R, I/32] (or [R, 2I/32], lo blocks after the hi blocks) and to GEMM2's
// per-tile layout (row r's expert from its (token, slot), its tile from the
// expert's plan; split: the lo byte kSfbLoOffset after the hi byte).  With
// `staged` (rows of at most kHqStageMaxI elements) the block's
// kHqStageRows rows come into shared memory by one bulk copy first, as in
// hquant_staged_kernel.
template <bool SPLIT>
__global__ void __launch_bounds__(256) hquant_mx_kernel(
    const __nv_bfloat16* __restrict__ h, int R, int I, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ token_slot, const int32_t* __restrict__ offsets,
    const int2* __restrict__ tile_plan, uint8_t* __restrict__ hq, uint8_t* __restrict__ h_sf,
    uint8_t* __restrict__ sfb, int staged, int32_t* __restrict__ status, uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t hstage[];
  __shared__ __align__(8) uint64_t bar;
  griddep_launch_dependents();   // as hquant_kernel: GEMM2 may start streaming weights
  const int r0 = blockIdx.x * kHqStageRows;
  const int nr = min(kHqStageRows, R - r0);
  if (staged) {
    // as hquant_staged_kernel: the block's rows by one bulk copy
    if (threadIdx.x == 0) {
      mbar_init(&bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
  }
  griddep_wait();
  if (staged) {
    if (threadIdx.x == 0) {
      const uint32_t bytes = static_cast<uint32_t>(nr) * static_cast<uint32_t>(I) * 2u;
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_load(hstage, h + static_cast<size_t>(r0) * I, bytes, &bar);
    }
    int32_t none = 0;
    if (!mbar_wait(&bar, 0, timeout_ns, status, kDevTimeout, &none)) return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = r0 + warp;
  if (warp >= nr) return;
  const int e = ids[token_slot[r]];
  const int64_t base = sfb_row_base(r, offsets[e], tile_plan[e], I / kTileK);
  const uint4* hr = staged
                        ? reinterpret_cast<const uint4*>(hstage) + static_cast<size_t>(warp) * I / 8
                        : reinterpret_cast<const uint4*>(h + static_cast<size_t>(r) * I);
  const int nblk = I / 32;
  const int64_t W = SPLIT ? 2 * I : I, nsf = SPLIT ? 2 * nblk : nblk;
  for (int b = lane; b < nblk; b += 32) {
    uint4 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = staged ? hr[4 * b + i] : __ldcg(hr + 4 * b + i);
    uint8_t sbyte, lbyte = 0;
    uint4 codes[2], lcodes[2];
    if constexpr (SPLIT)
      split_block(q, &sbyte, codes, &lbyte, lcodes);
    else
      mx_quant_block(q, &sbyte, codes);
    uint4* dst = reinterpret_cast<uint4*>(hq + r * W + 32 * b);
    dst[0] = codes[0];
    dst[1] = codes[1];
    h_sf[r * nsf + b] = sbyte;
    sfb[base + static_cast<int64_t>(b >> 2) * kSfbTileBytes + (b & 3)] = sbyte;
    if constexpr (SPLIT) {
      uint4* ldst = reinterpret_cast<uint4*>(hq + r * W + I + 32 * b);
      ldst[0] = lcodes[0];
      ldst[1] = lcodes[1];
      h_sf[r * nsf + nblk + b] = lbyte;
      sfb[base + static_cast<int64_t>(b >> 2) * kSfbTileBytes + kSfbLoOffset + (b & 3)] = lbyte;
    }
  }
}

// The top-k weighted combine [P4793 walkthrough: finalize fusion]: grid (T,
// ceil(H / 1024)); block (t, b) computes out[t, 1024 b .. 1024 b + 1023] =
// bf16( sum_j w[t, j] * y[row(t, j), c] ), float32 fused multiply-adds from 0
// in slot order j = 0 .. k-1, 8 columns (16 bytes) per thread.  The block's
// k row chunks (its 1024 columns of each of the token's k rows of y) come
// into shared memory by k bulk copies issued together, then are summed from
// there.  A timed-out wait for the copies records MOE_ERR_DEVICE_TIMEOUT.
__global__ void __launch_bounds__(128) combine_staged_kernel(
    const __nv_bfloat16* __restrict__ y, const float* __restrict__ wts,
    const int32_t* __restrict__ row_of, int k, int H, __nv_bfloat16* __restrict__ out,
    int32_t* __restrict__ status, uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t ystage[];   // [k][1024] bf16
  __shared__ int32_t rows[32];
  __shared__ float w[32];
  __shared__ __align__(8) uint64_t bar;
  const int t = blockIdx.x;
  // The row map and the routing weights come from the front end, which
  // finished before the previous kernel passed its wait (every kernel
  // signals its dependents only after its own wait), so they are read
  // before this grid's wait; y, the previous kernel's output, after it.
  if (static_cast<int>(threadIdx.x) < k) {
    rows[threadIdx.x] = __ldcg(row_of + static_cast<size_t>(t) * k + threadIdx.x);
    w[threadIdx.x] = __ldcg(wts + static_cast<size_t>(t) * k + threadIdx.x);
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();
  const int c0 = blockIdx.y * 1024;                       // first column
  const int ncol = min(1024, H - c0);                     // a multiple of 128
  const uint32_t bytes = static_cast<uint32_t>(ncol) * 2u;
  if (threadIdx.x < 32) {
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&bar, bytes * static_cast<uint32_t>(k));
    __syncwarp();
    if (static_cast<int>(threadIdx.x) < k)
      bulk_load(ystage + static_cast<size_t>(threadIdx.x) * 2048,
                y + static_cast<size_t>(rows[threadIdx.x]) * H + c0, bytes, &bar);
  }
  int32_t none = 0;
  if (!mbar_wait(&bar, 0, timeout_ns, status, kDevTimeout, &none)) return;
  const int i = threadIdx.x;   // the block's 16-byte vector
  if (8 * i >= ncol) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < k; ++j) {
    const uint4 q = reinterpret_cast<const uint4*>(ystage + static_cast<size_t>(j) * 2048)[i];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&q);
    const float wj = w[j];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 f = __bfloat1622float2(b[p]);
      acc[2 * p] = fmaf(wj, f.x, acc[2 * p]);
      acc[2 * p + 1] = fmaf(wj, f.y, acc[2 * p + 1]);
    }
  }
  uint4 r;
  __nv_bfloat162* rb = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
  for (int p = 0; p < 4; ++p) rb[p] = __floats2bfloat162_rn(acc[2 * p], acc[2 * p + 1]);
  reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H + c0)[i] = r;
}

// Waits on a barrier that nothing ever completes, with a bounded wait.
__global__ void timeout_selftest_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, timeout_ns, status, kDevTimeout, &abort_flag);
  __syncthreads();
}

}  // namespace

cudaError_t launch_hquant(const void* h, int R, int I, uint8_t* hq, float* h_scale,
                          int32_t* status, uint64_t timeout_ns, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  if (I <= kHqStageMaxI) {
    const size_t smem = static_cast<size_t>(kHqStageRows) * I * 2;
    static DeviceOnce smem_set;   // the limit for the longest staged row, once
    const cudaError_t e =
        set_smem_limit_once(hquant_staged_kernel, kHqStageRows * kHqStageMaxI * 2, smem_set);
    if (e != cudaSuccess) return e;
    return launch_pdl(hquant_staged_kernel, dim3((R + kHqStageRows - 1) / kHqStageRows),
                      dim3(32 * kHqStageRows), smem, s, static_cast<const __nv_bfloat16*>(h), R,
                      I, hq, h_scale, status, timeout_ns);
  }
  const int blocks = (R + 7) / 8;
  return launch_pdl(hquant_kernel, dim3(blocks), dim3(256), 0, s,
                    static_cast<const __nv_bfloat16*>(h), R, I, hq, h_scale);
}

cudaError_t launch_hquant_mx(int act, const void* h, int R, int I, const int32_t* ids,
                             const int32_t* token_slot, const int32_t* offsets,
                             const int2* tile_plan, uint8_t* hq, uint8_t* h_sf, uint8_t* sfb,
                             int32_t* status, uint64_t timeout_ns, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const int blocks = (R + kHqStageRows - 1) / kHqStageRows;
  auto kern = act == kActSplit ? hquant_mx_kernel<true> : hquant_mx_kernel<false>;
  const bool staged = I <= kHqStageMaxI;
  static DeviceOnce smem_set[2];   // the limit for the longest staged row, once
  const cudaError_t e = set_smem_limit_once(kern, kHqStageRows * kHqStageMaxI * 2,
                                            smem_set[act == kActSplit ? 1 : 0]);
  if (e != cudaSuccess) return e;
  const size_t smem = staged ? static_cast<size_t>(kHqStageRows) * I * 2 : 0;
  return launch_pdl(kern, dim3(blocks), dim3(32 * kHqStageRows), smem, s,
                    static_cast<const __nv_bfloat16*>(h), R, I, ids, token_slot, offsets,
                    tile_plan, hq, h_sf, sfb, staged ? 1 : 0, status, timeout_ns);
}

cudaError_t launch_combine(const void* y, const float* wts, const int32_t* row_of, int T, int k,
                           int H, void* out, int32_t* status, uint64_t timeout_ns,
                           cudaStream_t s) {
  const int nvec = H / 8;
  const size_t smem = static_cast<size_t>(k) * 2048;   // <= 64 KB (k <= 32)
  static DeviceOnce smem_set;
  const cudaError_t e = set_smem_limit_once(combine_staged_kernel, 32 * 2048, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(combine_staged_kernel, dim3(T, (nvec + 127) / 128), dim3(128), smem, s,
                    static_cast<const __nv_bfloat16*>(y), wts, row_of, k, H,
                    static_cast<__nv_bfloat16*>(out), status, timeout_ns);
}

cudaError_t launch_timeout_selftest(int32_t* status, uint64_t timeout_ns, cudaStream_t s) {
  timeout_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace moe
