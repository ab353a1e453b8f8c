/*
 * moe.h -- C ABI of the GB300 (sm_103a) fused MXFP4 x FP8 mixture-of-experts
 * forward.
 *
 * Pages cited (title and section):
 *   [P3738] flashinfer PR #3738, "perf: optimize MXFP4xBF16 & INT4xFP8 and add
 *           MXFP4xFP8 CUTLASS MoE backend for SM90": Description (runtime
 *           activation expansion and per-token FP8 activation quantization;
 *           precomputed grouped GEMM work scheduling and TMA descriptor state;
 *           folded weight-scale storage; per-token scale epilogue),
 *           Implementation Notes, review comments (interleave preconditions
 *           n % 16 and k % 64; K % 32 for the scale shape; zero routed tokens
 *           must be a no-op, not an error).
 *   [P4411] flashinfer PR #4411, "revert(moe): revert #3738 SM90 CUTLASS MoE
 *           backend (+ dependents #4025, #4080) on release-v0.6.17":
 *           Description (caller-owned workspace and its size query kept as
 *           public API; a null TMA descriptor corrupts the CUDA context).
 *   [P4793] flashinfer PR #4793, "Unify MoE CuTe DSL dispatch to be dtype
 *           agnostic": review comments (uint8 scale tensors; quant_mode
 *           strings "w4a4"/"w4a8"; fail fast with NotImplementedError on
 *           unsupported architectures).
 *   [P3614] flashinfer PR #3614, "fix: make the cutlass MoE gemm profiler
 *           MXFP8-aware": description (never launch with a null scale-factor
 *           buffer; fail fast with 'No valid tactics' instead of a deep
 *           kernel assert).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless the name says host.  The
 *     caller owns all memory; no entry point allocates device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; the return value reports only
 *     host-side validation and launch errors.  Device-side errors (a bounded
 *     wait that ran out) are written to a status word in the workspace and
 *     read back with moe_read_device_status().
 *   - No C++ exception crosses the ABI.  Invalid arguments are rejected before
 *     any CUDA call is made.
 *   - num_tokens == 0 returns MOE_OK and launches nothing [P3738 review
 *     comments: an empty routed batch is a no-op].
 */
#ifndef PRECISION_MOE_GROUPED_GB300_MOE_H_
#define PRECISION_MOE_GROUPED_GB300_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,        /* null pointer, negative size, bad enum   */
  MOE_ERR_UNSUPPORTED = -2,        /* mode/shape/device the library cannot run */
  MOE_ERR_MISALIGNED = -3,         /* pointer alignment or shape divisibility */
  MOE_ERR_WORKSPACE_TOO_SMALL = -4,
  MOE_ERR_CUDA = -5,               /* a CUDA runtime/driver call failed       */
  MOE_ERR_DEVICE_TIMEOUT = -6,     /* a device-side bounded wait ran out      */
  MOE_ERR_DEVICE_CHECK = -7        /* checked builds (libmoe_checked.so, built
                                      with MOE_CHECKS) only: a device-side
                                      bounds check of the work map failed    */
} moe_status;

/* Quantisation modes (the pages' W4A8 / W4A16 / MXFP8 paths); all three are
 * implemented. */
typedef enum {
  MOE_W4A8_MXFP4_FP8 = 0,    /* MXFP4 weights, runtime per-token FP8 E4M3 acts */
  MOE_W4A16_MXFP4_BF16 = 1,  /* MXFP4 weights, bf16 activations (computed on
                                the FP8 tensor cores as two MXFP8 terms per
                                activation: exact for every element within
                                2^13 of its 32-block's maximum)           */
  MOE_W8A8_MXFP8 = 2         /* MXFP8 weights and MXFP8 activations           */
} moe_quant_mode;

/* Problem shape.  Activation SwiGLU and softmax-top-k-renormalised routing
 * are fixed.  Limits: num_tokens >= 0; 1 <= num_experts <= 1024;
 * 1 <= top_k <= min(num_experts, 32); hidden and inter positive multiples of
 * 128; num_tokens * top_k < 2^31; num_experts * 2 * inter * hidden / 128 <
 * 2^31 (the GEMMs' 32-bit weight-box coordinates) and
 * (T*k/16 + min(E, T*k) + 1) * max(2*inter, hidden) / 128 < 2^31 (their
 * work-item counters); MOE_ERR_UNSUPPORTED otherwise. */
typedef struct {
  int32_t num_tokens;   /* T */
  int32_t num_experts;  /* E */
  int32_t top_k;        /* k */
  int32_t hidden;       /* H */
  int32_t inter;        /* I (w1 has 2I rows: gate rows 0..I-1, up rows I..2I-1) */
} moe_shape;

/* Kernels one forward launches, in stream order: route, scan, rank,
 * quant_scatter, gemm1, hquant, gemm2, combine (moe_stage_name() names them).
 * The scatter kernel ranks the expanded rows itself, so the "rank" stage is
 * empty and a large batch launches 7 kernels.  For num_tokens <=
 * MOE_SMALL_BATCH_TOKENS the expansion (scan, rank, quant_scatter) runs as
 * one kernel, timed as stage "scan"; the "quant_scatter" stage is then empty
 * too and the forward launches 6 kernels.
 * For num_tokens <= MOE_TINY_BATCH_TOKENS in the W4A8 mode routing and
 * expansion run as one kernel, timed as stage "route" (5 kernels).
 * Kernels are launched with programmatic dependent launch: each may start
 * while its predecessor finishes and waits for the predecessor's results. */
#define MOE_NUM_STAGES 8
#define MOE_SMALL_BATCH_TOKENS 256
#define MOE_TINY_BATCH_TOKENS 32

/* Optional per-call settings (moe_forward_ex); zero-initialise for defaults. */
typedef struct {
  int32_t tile_variant;  /* 0 auto (3 while experts average <= 8 rows, 1 up
                            to 32, else 5); 1 decode tiles (<= 32 tokens per
                            GEMM tile, 10-stage weight pipeline); 2 prefill
                            tiles (<= 224); 3 decode tiles of <= 16 tokens
                            (12 stages); 4 prefill tiles with two MMA
                            issuers; 5 tiles of <= 160 tokens with a 6-stage
                            pipeline; 6 tiles of <= 160 tokens on CTA pairs
                            (two SMs share each 256-row MMA; W4A8 with
                            hidden a multiple of 256 -- otherwise the GEMM
                            runs as 5)                                    */
  int32_t timeout_ms;    /* device bounded-wait limit, 0 = 1000 ms           */
  void* stage_events;    /* NULL, or an array of MOE_NUM_STAGES + 1 cudaEvent_t
                            (caller-created): event 0 is recorded on `stream`
                            before the first kernel and event i right after
                            kernel i, so event pairs time each kernel      */
  int32_t prefetch_stages; /* L2 prefetch distance of the GEMM weight stream,
                            in K stages: 0 = default (off), < 0 = off   */
  int32_t gather_x;      /* W4A8 batches of more than MOE_SMALL_BATCH_TOKENS
                            tokens with x in device memory, tile variants
                            1-5: 1 = the expansion writes each token's FP8
                            row once (token-major [T, H] in the xq region;
                            the x_scale of every expanded row as before)
                            and GEMM1's producers gather each tile's rows
                            by token with asynchronous copies; 0 or -1 =
                            the expanded [R, H] copy (the default: faster
                            from T = 2048 on).  Ignored elsewhere.       */
  int32_t fuse_combine;  /* tile variants 1-5: 1 = GEMM2's epilogue also
                            forms the weighted top-k combine (the last of a
                            token's k slots to finish a 32-column segment
                            sums the k rows of y in slot order, the
                            combine kernel's arithmetic, and writes out),
                            no combine kernel; 0 or -1 = the combine
                            kernel (the default: faster at every size
                            measured, e.g. DSV3 T=4096 1.50 against
                            3.50 ms).                                   */
  int32_t reserved[1];   /* must be zero                                     */
} moe_options;

/* Byte offsets of the intermediate tensors inside the workspace, for tests
 * and diagnostics (R = num_tokens * top_k expanded rows).  Layouts:
 *   status      int32[4]      status word, tile count, R and E (checked builds; else spare)
 *   ids         int32[T,k]    routed expert of (token, slot), descending logit
 *   weights     float[T,k]    renormalised softmax routing weights
 *   row_of      int32[T,k]    expanded row of (token, slot)
 *   counts      int32[E]      rows per expert
 *   offsets     int32[E+1]    exclusive scan of counts
 *   token_slot  int32[R]      token*top_k + slot of each expanded row
 *   tiles       int32[4*max]  GEMM work map: (expert, first row, rows, 0)
 *   xq          uint8[R,H]    FP8 E4M3 codes of the expanded activations
 *                             (W4A16: uint8[R,2H], the hi terms in columns
 *                             0..H-1, the lo terms -- hi's exact residual
 *                             -- in H..2H-1)
 *   x_scale     float[R]      per-row (per-token) activation scale
 *   h           bf16[R,I]     SwiGLU output
 *   hq          uint8[R,I]    FP8 E4M3 codes of h (W4A16: uint8[R,2I], hi | lo)
 *   h_scale     float[R]      per-row scale of hq
 *   y           bf16[R,H]     GEMM2 output (scaled)
 *   x_stage, logits_stage, out_stage: device staging used by moe_forward_host
 *   tile_plan   int32[E,2]    per expert: first GEMM tile, rows per tile
 * MXFP8 (W8A8) and W4A16 only (0 bytes otherwise; x_scale / h_scale unused):
 *   x_sf        uint8[R,H/32] E8M0 block scales of xq, row-major (W4A16:
 *                             [R,2H/32], the hi blocks then the lo blocks)
 *   h_sf        uint8[R,I/32] E8M0 block scales of hq, row-major (W4A16:
 *                             [R,2I/32])
 *   x_sf_tiled, h_sf_tiled    the same scales in the GEMMs' per-tile layout:
 *                             1024 bytes per (tile, 128-K stage)
 * The workspace ends with int32 [T, H/128, 4] arrival counters used by
 * moe_options.fuse_combine (cleared by the forward's first kernel). */
typedef struct {
  uint64_t status, ids, weights, row_of, counts, offsets, chunk_counts, token_slot,
      tiles, xq, x_scale, h, hq, h_scale, y, x_stage, logits_stage, out_stage, tile_plan,
      x_sf, h_sf, x_sf_tiled, h_sf_tiled, total;
  int32_t max_tiles, num_chunks, reserved[6];
} moe_ws_layout;

/* Workspace bytes moe_forward needs for `shape` and `quant_mode` (host-only,
 * pure).  Returns 0 for an invalid shape or mode.  The caller allocates it
 * (256-byte aligned) [P4411 Description: caller-owned workspace and its size
 * query]. */
size_t moe_workspace_size(const moe_shape* shape, int32_t quant_mode);

/* Fills `layout` with the workspace carving used by moe_forward. */
int32_t moe_workspace_layout(const moe_shape* shape, int32_t quant_mode,
                             moe_ws_layout* layout);

/* Re-lays the expert weights from the user layout into the layout the GEMM
 * kernels stream (bit-preserving: only rows and scale bytes move)
 * [P3738 Description: folded weight-scale storage independent of the tile
 * choice; review comments: interleave kernels and their n % 16, k % 64
 * preconditions].
 * User layout (W4A8 / W4A16), all uint8, device:
 *   w1    [E, 2I, H/2]  E2M1 codes, two per byte, low nibble = even k
 *   w1_sf [E, 2I, H/32] E8M0 scale per 32 consecutive k
 *   w2    [E, H, I/2],  w2_sf [E, H, I/32]
 * User layout (W8A8, MXFP8 [P3614]): w1 [E, 2I, H] and w2 [E, H, I] hold one
 * E4M3 code per byte; w1_sf and w2_sf are as above.
 * Outputs have the same byte sizes and must not alias the inputs.  Pointers
 * must be 256-byte aligned.  Asynchronous on `stream`. */
int32_t moe_prepare_weights(const moe_shape* shape, int32_t quant_mode,
                            const void* w1, const void* w1_sf, const void* w2,
                            const void* w2_sf, void* w1_p, void* w1_sf_p, void* w2_p,
                            void* w2_sf_p, void* stream);

/* The fused forward: routing -> expert-sorted expansion with per-token FP8
 * quantisation -> GEMM1 (gate|up) with SwiGLU and the token scale in its
 * epilogue -> per-row FP8 quantisation of h -> GEMM2 -> top-k weighted
 * combine.
 *   x              bf16  [T, H]  (16-byte aligned)
 *   router_logits  float [T, E]  finite values (a NaN is ranked as -inf, so
 *                                 the routed ids stay in range; it gets
 *                                 weight 0 unless the whole row is NaN or
 *                                 -inf, which gives NaN weights)
 *   w1_p .. w2_sf_p              prepared weights (moe_prepare_weights)
 *   out            bf16  [T, H]  written in full (16-byte aligned)
 *   workspace      >= moe_workspace_size() bytes, 256-byte aligned
 * [P3738 Description, Implementation Notes]. */
int32_t moe_forward(const moe_shape* shape, int32_t quant_mode, const void* x,
                    const float* router_logits, const void* w1_p, const void* w1_sf_p,
                    const void* w2_p, const void* w2_sf_p, void* out, void* workspace,
                    size_t workspace_bytes, void* stream);

/* moe_forward with options (opts may be NULL). */
int32_t moe_forward_ex(const moe_shape* shape, int32_t quant_mode, const void* x,
                       const float* router_logits, const void* w1_p, const void* w1_sf_p,
                       const void* w2_p, const void* w2_sf_p, void* out, void* workspace,
                       size_t workspace_bytes, void* stream, const moe_options* opts);

/* End-to-end variant with HOST activations x_host (bf16 [T,H]), logits_host
 * (float [T,E]) and out_host (bf16 [T,H]), all on `stream`.  A page-locked
 * host buffer (cudaHostAlloc, cudaMallocHost, cudaHostRegister) is read or
 * written in place by the kernels, over the host link, so its transfer
 * overlaps the computation; any other host buffer is copied through the
 * workspace's staging area (x and logits before the forward, out after it).
 * Host buffers must stay valid, and out_host unread, until the stream
 * reaches this point.  The results are the same either way. */
int32_t moe_forward_host(const moe_shape* shape, int32_t quant_mode, const void* x_host,
                         const float* logits_host, const void* w1_p, const void* w1_sf_p,
                         const void* w2_p, const void* w2_sf_p, void* out_host,
                         void* workspace, size_t workspace_bytes, void* stream,
                         const moe_options* opts);

/* Workspace bytes moe_forward_host_steps needs: moe_workspace_size plus a
 * second staging set (x, logits and out of one step).  0 for an invalid
 * shape or mode. */
size_t moe_steps_workspace_size(const moe_shape* shape, int32_t quant_mode);

/* n_steps forwards of one shape, step i from host buffers x_host[i] (bf16
 * [T,H]), logits_host[i] (float [T,E]) into out_host[i] (bf16 [T,H]), with
 * the host<->device copies overlapped with the computation: two copy
 * streams of its own move step i+1's inputs into one device staging set and
 * step i-1's output out of the other while step i computes on `stream`
 * (double-buffered staging; the first set is the workspace's x_stage /
 * logits_stage / out_stage, the second follows the moe_workspace_size bytes).
 * The overlap needs page-locked host buffers (cudaHostAlloc,
 * cudaMallocHost, cudaHostRegister); others are copied synchronously by the
 * runtime.  Each step's results equal moe_forward's on the same inputs
 * [P3738 Description: the fused MoE forward; P4411 Description:
 * caller-owned workspace].
 *   workspace: device, 256-byte aligned, >= moe_steps_workspace_size bytes
 *   opts: as moe_forward_ex; stage_events must be NULL (MOE_ERR_INVALID_ARG)
 * Asynchronous: returns once everything is queued; `stream` reaches its end
 * when every out_host[i] is written.  Host buffers must stay valid, and the
 * outputs unread, until then.  Errors: the argument errors of moe_forward,
 * n_steps < 0 or a NULL step pointer (MOE_ERR_INVALID_ARG), a workspace
 * below moe_steps_workspace_size (MOE_ERR_WORKSPACE_TOO_SMALL); a CUDA error
 * while queueing returns MOE_ERR_CUDA with the steps before it queued. */
int32_t moe_forward_host_steps(const moe_shape* shape, int32_t quant_mode, int32_t n_steps,
                               const void* const* x_host, const float* const* logits_host,
                               const void* w1_p, const void* w1_sf_p, const void* w2_p,
                               const void* w2_sf_p, void* const* out_host, void* workspace,
                               size_t workspace_bytes, void* stream, const moe_options* opts);

/* Reads the device status word of `workspace` (synchronises `stream`).
 * *status = MOE_OK or the moe_status of the first device-side error since
 * the workspace was last used by moe_forward (which clears it). */
int32_t moe_read_device_status(const void* workspace, void* stream, int32_t* status);

/* Exercises the bounded-wait machinery: launches one block that waits on a
 * barrier nothing completes, with a limit of `timeout_us`; the wait gives
 * up, writes MOE_ERR_DEVICE_TIMEOUT to the status word of `workspace` and
 * the kernel returns normally.  For tests of the failure path. */
int32_t moe_selftest_timeout(void* workspace, int32_t timeout_us, void* stream);

/* Size of the static device scratch moe_route_noalloc uses (4 MiB). */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)

/* Routing front end without any caller-provided scratch: top-k softmax
 * routing, per-expert offsets and the expert-major row map -- the same
 * kernels and results as the first stages of moe_forward -- for callers that
 * cannot allocate device memory.  Examples: a plugin inside an inference
 * server that is handed only its input and output buffers and has no
 * allocator of its own, or a latency-critical path that must not call
 * cudaMalloc after start-up (it can synchronise the device and take
 * unbounded time).  The flashinfer PRs have no counterpart to it.
 *   router_logits  float [T, E] (device)      input
 *   ids            int32 [T, k] (device)      output: experts, descending logit
 *   weights        float [T, k] (device)      output: renormalised weights
 *   offsets        int32 [E + 1] (device)     output: exclusive scan of counts
 *   row_of         int32 [T, k] (device)      output: expert-major row of (t, j)
 * Its scratch is one file-scope device array of MOE_NOALLOC_SCRATCH_BYTES,
 * which every GPU that loads this library holds until the process exits.
 * Shapes needing more (about (T/32)*E*4 + T*k*4.5 + E*20 bytes) are rejected
 * with MOE_ERR_WORKSPACE_TOO_SMALL and a message in moe_last_error().  The
 * first call in each CUDA context looks up the array's device address (with
 * that context current) and caches it under the context's process-unique
 * id; make that first call before any stream capture.  All
 * calls share the one array, which keeps the last call's contents (every
 * word a call reads is written earlier in the same call): calls that overlap
 * on the GPU -- on different streams or from different host threads -- race
 * on it and must be serialised.  Allocates nothing (no cudaMalloc/cudaFree).
 * Runs on sm_103a devices only (MOE_ERR_UNSUPPORTED elsewhere, as
 * moe_forward).  num_tokens == 0 returns MOE_OK, launches nothing and leaves
 * every output untouched (the offsets of an empty batch are all zero; a
 * caller that reads them must write those zeros itself). */
int32_t moe_route_noalloc(const moe_shape* shape, const float* router_logits, int32_t* ids,
                          float* weights, int32_t* offsets, int32_t* row_of, void* stream);

/* Message describing the last error returned on the calling thread. */
const char* moe_last_error(void);

/* Name of forward kernel `stage` (0 .. MOE_NUM_STAGES-1), or NULL. */
const char* moe_stage_name(int32_t stage);

/* Static description of a status code. */
const char* moe_status_string(int32_t status);

/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* PRECISION_MOE_GROUPED_GB300_MOE_H_ */
