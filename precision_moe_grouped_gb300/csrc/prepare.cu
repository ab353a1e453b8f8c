// prepare.cu -- one-time re-layout of the expert weights for the GEMM kernels
// (bit-preserving: rows and scale bytes move, no value changes).
//
// Pages cited (title and section):
//   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
//           MXFP4xFP8 CUTLASS MoE backend for SM90": Description ("use folded
//           weight-scale storage so the weight-scale layout is independent of
//           the profiled TileK"), review comments (weight interleave kernels
//           work on 16-row x 64-K groups and need n % 16 == 0, k % 64 == 0).
//
// Layouts produced (per expert e, M rows of weights, K reduction elements):
//   * weights: blocked into contiguous boxes, one per (e, M-tile mt,
//     K-stage ks of 128 elements): box ((e * MT + mt) * KS + ks) holds tile
//     rows 0..127 of that K range, 64 bytes (128 packed E2M1 codes) per row
//     -- 8 KB boxes -- or, for the MXFP8 weights of the W8A8 mode, 128 bytes
//     (128 E4M3 codes) per row -- 16 KB boxes.
//     A GEMM work item then streams one contiguous run of KS boxes, and every
//     TMA box load is a single 8 KB read.  GEMM1's w1 rows are also permuted
//     so that every 128-row M-tile holds 64 gate rows and the 64 matching up
//     rows, interleaved in groups of 16: tile row 32q + i is gate feature
//     64*mt + 16q + i for i < 16 and up feature 64*mt + 16q + (i - 16) for
//     i >= 16.  The GEMM1 epilogue then pairs gate and up of one feature
//     across lanes i and i+16 of the same warp.  GEMM2's w2 rows keep their
//     order.
//   * scales: for each (e, mt, ks) one 512-byte block laid out as 32 x 16
//     bytes: bytes [16l + 4i, 16l + 4i + 4) are the four E8M0 bytes (K-blocks
//     4ks .. 4ks+3) of tile row 32i + l.  This is the 32-lane x 128-bit shape
//     tcgen05.cp copies into TMEM with 4-way lane-quarter replication; the
//     block-scaled MMA then reads row m's scale from TMEM lane m, column
//     m/32, byte = the scale-factor id.
#include "moe_internal.h"

namespace moe {

namespace {

__host__ __device__ inline int w1_src_row(int p, int I) {
  const int mt = p / 128, r = p % 128, q = r / 32, i = r % 32;
  const int f = 64 * mt + 16 * q + (i & 15);
  return i < 16 ? f : I + f;
}

// One thread per destination 16-byte vector of the blocked weight layout;
// VPR = 16-byte vectors per box row (4: 128 packed E2M1 codes, 8: 128 E4M3
// codes).
template <int VPR>
__global__ void block_weights_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                     int64_t total_vec, int M, int K, int swiglu_I) {
  const int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (v >= total_vec) return;
  const int KS = K / 128, MT = M / 128;
  const int q = static_cast<int>(v % VPR);              // 16-byte piece of a box row
  const int r = static_cast<int>((v / VPR) & 127);      // box row
  const int64_t blk = v / (VPR * 128);                  // (e * MT + mt) * KS + ks
  const int ks = static_cast<int>(blk % KS);
  const int64_t emt = blk / KS;
  const int mt = static_cast<int>(emt % MT);
  const int64_t e = emt / MT;
  const int p = mt * 128 + r;
  const int srow = swiglu_I > 0 ? w1_src_row(p, swiglu_I) : p;
  const int64_t vec_per_row = static_cast<int64_t>(K / 128) * VPR;
  dst[v] = src[(e * M + srow) * vec_per_row + ks * VPR + q];
}

// One thread per destination 32-bit word.
__global__ void sf_layout_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst,
                                 int64_t total_words, int M, int K, int swiglu_I) {
  const int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (w >= total_words) return;
  const int KS = K / 128, MT = M / 128;
  const int words_per_row = K / 128;  // 4 scale bytes per 128 K elements
  const int i = static_cast<int>(w & 3);
  const int l = static_cast<int>((w >> 2) & 31);
  const int64_t blk = w >> 7;  // (e * MT + mt) * KS + ks
  const int ks = static_cast<int>(blk % KS);
  const int64_t emt = blk / KS;
  const int mt = static_cast<int>(emt % MT);
  const int64_t e = emt / MT;
  const int p = mt * 128 + 32 * i + l;
  const int srow = swiglu_I > 0 ? w1_src_row(p, swiglu_I) : p;
  dst[w] = src[(e * M + srow) * words_per_row + ks];
}

}  // namespace

cudaError_t launch_prepare(const uint8_t* w, const uint8_t* sf, uint8_t* w_p, uint8_t* sf_p,
                           int E, int M, int K, int swiglu_I, bool fp8, cudaStream_t s) {
  const int vpr = fp8 ? 8 : 4;
  const int64_t vecs = static_cast<int64_t>(E) * M * (K / 128) * vpr;
  auto kern = fp8 ? block_weights_kernel<8> : block_weights_kernel<4>;
  kern<<<static_cast<unsigned>((vecs + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(w), reinterpret_cast<uint4*>(w_p), vecs, M, K, swiglu_I);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int64_t words = static_cast<int64_t>(E) * M * (K / 128);
  sf_layout_kernel<<<static_cast<unsigned>((words + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const uint32_t*>(sf), reinterpret_cast<uint32_t*>(sf_p), words, M, K,
      swiglu_I);
  return cudaGetLastError();
}

}  // namespace moe
