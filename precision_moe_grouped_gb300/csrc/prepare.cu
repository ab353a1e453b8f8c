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
//   * weight rows: GEMM1's w1 rows are permuted so that every 128-row M-tile
//     holds 64 gate rows and the 64 matching up rows, interleaved in groups
//     of 16: tile row 32q + i is gate feature 64*mt + 16q + i for i < 16 and
//     up feature 64*mt + 16q + (i - 16) for i >= 16.  The GEMM1 epilogue then
//     pairs gate and up of one feature across lanes i and i+16 of the same
//     warp.  GEMM2's w2 rows keep their order.
//   * scales: for each (e, M-tile mt, K-stage ks of 128 elements) one 512-byte
//     block laid out as 32 x 16 bytes: bytes [16l + 4i, 16l + 4i + 4) are the
//     four E8M0 bytes (K-blocks 4ks .. 4ks+3) of tile row 32i + l.  This is
//     the 32-lane x 128-bit shape tcgen05.cp copies into TMEM with 4-way
//     lane-quarter replication; the block-scaled MMA then reads row m's scale
//     from TMEM lane m, column m/32, byte = the scale-factor id.
#include "moe_internal.h"

namespace moe {

namespace {

__host__ __device__ inline int w1_src_row(int p, int I) {
  const int mt = p / 128, r = p % 128, q = r / 32, i = r % 32;
  const int f = 64 * mt + 16 * q + (i & 15);
  return i < 16 ? f : I + f;
}

__global__ void permute_w1_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                       int rows_per_expert, int vec_per_row, int I) {
  const int64_t row = blockIdx.x;  // e * rows_per_expert + p
  const int e = static_cast<int>(row / rows_per_expert);
  const int p = static_cast<int>(row % rows_per_expert);
  const int64_t srow = static_cast<int64_t>(e) * rows_per_expert + w1_src_row(p, I);
  for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x)
    dst[row * vec_per_row + v] = src[srow * vec_per_row + v];
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

cudaError_t launch_prepare_w1(const uint8_t* w1, const uint8_t* w1_sf, uint8_t* w1_p,
                              uint8_t* w1_sf_p, int E, int I, int H, cudaStream_t s) {
  const int M = 2 * I;
  const int vec_per_row = (H / 2) / 16;
  permute_w1_rows_kernel<<<static_cast<unsigned>(static_cast<int64_t>(E) * M), 128, 0, s>>>(
      reinterpret_cast<const uint4*>(w1), reinterpret_cast<uint4*>(w1_p), M, vec_per_row, I);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int64_t words = static_cast<int64_t>(E) * M * (H / 128);
  sf_layout_kernel<<<static_cast<unsigned>((words + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const uint32_t*>(w1_sf), reinterpret_cast<uint32_t*>(w1_sf_p), words, M,
      H, I);
  return cudaGetLastError();
}

cudaError_t launch_prepare_sf_plain(const uint8_t* sf, uint8_t* sf_p, int E, int M, int K,
                                    cudaStream_t s) {
  const int64_t words = static_cast<int64_t>(E) * M * (K / 128);
  sf_layout_kernel<<<static_cast<unsigned>((words + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const uint32_t*>(sf), reinterpret_cast<uint32_t*>(sf_p), words, M, K, 0);
  return cudaGetLastError();
}

}  // namespace moe
