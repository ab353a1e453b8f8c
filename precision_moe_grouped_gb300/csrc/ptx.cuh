// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers with bounded
// waits, TMA (tensor and bulk copies), and the tcgen05 tensor-core family
// (TMEM allocation, smem->TMEM copies, block-scaled MMA, TMEM loads).
//
// Every wait here is bounded by a wall-clock limit (%globaltimer, ns).  When
// the limit passes, the wait records an error code in the caller's status
// word and returns false; callers then leave their loops, so a kernel never
// spins forever.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace moe {

// ---------------------------------------------------------------- basics
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool elect_lane0() { return (threadIdx.x & 31) == 0; }

// ------------------------------------------------------ programmatic launch
// Every kernel of the forward is launched with programmatic stream
// serialisation: it may start while its predecessor finishes, so it waits
// for the predecessor's results here before reading them, and lets its own
// successor start launching as early as possible.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the thread sleep until the phase completes or
// `suspend_ns` pass (the hardware wakes it on completion), so waiting warps
// do not take issue slots from the warps doing work.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar_addr, uint32_t parity,
                                                      uint32_t suspend_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}

// Longest sleep of one suspended try_wait: the abort flag and the wall-clock
// limit are checked between sleeps.
constexpr uint32_t kSuspendNs = 20000;

// Waits until the phase with parity `parity` of `bar` has completed, at most
// `timeout_ns`; also gives up early when *abort is set by another role.  On
// giving up it records `code` in *status (first error wins) and sets *abort.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          int32_t* status, int32_t code,
                                          volatile int32_t* abort) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_suspend(a, parity, kSuspendNs)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      atomicCAS(status, 0, code);
      *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled TMA load into shared memory, completing on `bar` (tx bytes).
// c0 is the innermost coordinate (elements), c1 the row.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* m, int32_t c0,
                                            int32_t c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 under L2 cache
// policy `pol` (both addresses 16-byte aligned), and the arrival on `bar`
// once this thread's earlier such copies have completed (counted in the
// barrier's expected arrivals).  The policies: evict-last (lines to keep)
// and evict-first (lines read once); tma_load_2d under a policy.
__device__ __forceinline__ void cp_async_16_hint(void* smem_dst, const void* gsrc, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(gsrc)), "l"(pol)
               : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* m, int32_t c0,
                                                 int32_t c1, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Prefetch a 2-D tile of a tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* m, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1)
               : "memory");
}

// Prefetch `bytes` (multiple of 16) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                   reinterpret_cast<uint64_t>(gsrc)),
               "r"(bytes)
               : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation by one full warp; the base address is written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` once every tcgen05 async operation issued so far by this
// thread (MMAs and smem->TMEM copies) has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Warp-wide forms: the whole warp executes the call with identical
// arguments and one elected lane issues the instruction.  Keeping the issue
// loop warp-uniform (instead of running it in lane 0 alone) measured ~30%
// fewer cycles per issued stage on sm_103a.
__device__ __forceinline__ void tc_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// All lanes wait (bounded) and agree on the outcome, so a loop that breaks
// on failure stays warp-uniform.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity,
                                               uint64_t timeout_ns, int32_t* status, int32_t code,
                                               volatile int32_t* abort) {
  const bool ok = mbar_wait(bar, parity, timeout_ns, status, code, abort);
  return __all_sync(0xffffffffu, ok);
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), fixed version bits 46-47 = 1, layout
// type in bits 61-63 (0 = no swizzle, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(layout & 7) << 61;
  return d;
}

// Copy a 32-row x 128-bit matrix from shared memory into TMEM and repeat it
// in all four 32-lane quarters (the scale-factor staging shape).
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// One 128-K pipeline stage from one elected lane, in a single block so that
// the warp elects once: the weight scales into TMEM (32x128b.warpx4 from
// sfa_src), the 4 block-scaled MMAs of K sub-steps 0..3 (A and B advanced
// 32 bytes per step; scale IDs = the step; the first accumulates only when
// acc0 != 0), and a commit to the stage's empty barrier.
__device__ __forceinline__ void tc_stage_mx4_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                  uint32_t id0, uint32_t sfa_tmem,
                                                  uint64_t sfa_src, uint32_t sfb_tmem,
                                                  uint32_t acc0, uint32_t empty_bar) {
  asm volatile(
      "{\n\t.reg .pred e, p, q;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %7, 0;\n\t"
      "setp.eq.b32 q, %7, %7;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%4], %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%6], p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %9, %10, %11, [%4], [%6], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %12, %13, %14, [%4], [%6], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %15, %16, %17, [%4], [%6], q;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%8];\n\t}" ::
          "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(id0), "r"(sfa_tmem), "l"(sfa_src),
      "r"(sfb_tmem), "r"(acc0), "r"(empty_bar),
      "l"(adesc + 2), "l"(bdesc + 2), "r"(id0 | (1u << 4) | (1u << 29)),
      "l"(adesc + 4), "l"(bdesc + 4), "r"(id0 | (2u << 4) | (2u << 29)),
      "l"(adesc + 6), "l"(bdesc + 6), "r"(id0 | (3u << 4) | (3u << 29))
      : "memory");
}

// As tc_stage_mx4_warp, with per-stage activation scales (MXFP8): after the
// weight scales, the activation scales into TMEM from sfb_src (and the next
// 512 bytes into sfb_tmem + 4 when sfb2 != 0: MMA-N > 128), then the 4 MMAs
// and the commit.
__device__ __forceinline__ void tc_stage_mx4_sfb_warp(uint32_t d_tmem, uint64_t adesc,
                                                      uint64_t bdesc, uint32_t id0,
                                                      uint32_t sfa_tmem, uint64_t sfa_src,
                                                      uint32_t sfb_tmem, uint64_t sfb_src,
                                                      uint32_t sfb2, uint32_t acc0,
                                                      uint32_t empty_bar) {
  asm volatile(
      "{\n\t.reg .pred e, e2, p, q;\n\t"
      ".reg .b64 a1, a2, a3, b1, b2, b3, s2;\n\t"
      ".reg .b32 i1, i2, i3, t2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %9, 0;\n\t"
      "setp.eq.b32 q, %9, %9;\n\t"
      "setp.ne.and.b32 e2, %8, 0, e;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
      "or.b32 i1, %3, 0x20000010;\n\tor.b32 i2, %3, 0x40000020;\n\tor.b32 i3, %3, 0x60000030;\n\t"
      "add.s64 s2, %7, 32;\n\tadd.u32 t2, %6, 4;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%4], %5;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%6], %7;\n\t"
      "@e2 tcgen05.cp.cta_group::1.32x128b.warpx4 [t2], s2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%6], p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], a1, b1, i1, [%4], [%6], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], a2, b2, i2, [%4], [%6], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], a3, b3, i3, [%4], [%6], q;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n\t}" ::
          "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(id0), "r"(sfa_tmem), "l"(sfa_src),
      "r"(sfb_tmem), "l"(sfb_src), "r"(sfb2), "r"(acc0), "r"(empty_bar)
      : "memory");
}

// A split-activation stage (W4A16): weight scales, the hi term's scales
// (sfb_src) and the lo term's (the next 512 bytes, into sfb_tmem + 4), the 4
// MMAs of the hi box (bdesc; the first accumulates only when acc0 != 0) and
// the 4 of the lo box (bdesc_lo) into the same accumulator, and the commit.
__device__ __forceinline__ void tc_stage_split_warp(uint32_t d_tmem, uint64_t adesc,
                                                    uint64_t bdesc, uint64_t bdesc_lo,
                                                    uint32_t id0, uint32_t sfa_tmem,
                                                    uint64_t sfa_src, uint32_t sfb_tmem,
                                                    uint64_t sfb_src, uint32_t acc0,
                                                    uint32_t empty_bar) {
  asm volatile(
      "{\n\t.reg .pred e, p, q;\n\t"
      ".reg .b64 a1, a2, a3, b1, b2, b3, l1, l2, l3, s2;\n\t"
      ".reg .b32 i1, i2, i3, t2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %9, 0;\n\t"
      "setp.eq.b32 q, %9, %9;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
      "add.s64 l1, %3, 2;\n\tadd.s64 l2, %3, 4;\n\tadd.s64 l3, %3, 6;\n\t"
      "or.b32 i1, %4, 0x20000010;\n\tor.b32 i2, %4, 0x40000020;\n\tor.b32 i3, %4, 0x60000030;\n\t"
      "add.s64 s2, %8, 32;\n\tadd.u32 t2, %7, 4;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%5], %6;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%7], %8;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [t2], s2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %4, [%5], [%7], p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], a1, b1, i1, [%5], [%7], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], a2, b2, i2, [%5], [%7], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], a3, b3, i3, [%5], [%7], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %3, %4, [%5], [t2], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], a1, l1, i1, [%5], [t2], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], a2, l2, i2, [%5], [t2], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], a3, l3, i3, [%5], [t2], q;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n\t}" ::
          "r"(d_tmem), "l"(adesc), "l"(bdesc), "l"(bdesc_lo), "r"(id0), "r"(sfa_tmem),
      "l"(sfa_src), "r"(sfb_tmem), "l"(sfb_src), "r"(acc0), "r"(empty_bar)
      : "memory");
}

// Instruction descriptor for block-scaled .kind::mxf8f6f4, M = 128, both
// operands K-major, E8M0 scales.  Formats: 0 = E4M3, 5 = E2M1.
__host__ __device__ constexpr uint32_t idesc_mx(uint32_t a_fmt, uint32_t b_fmt, uint32_t n,
                                                uint32_t a_sf_id, uint32_t b_sf_id) {
  return (b_sf_id << 4) | (a_fmt << 7) | (b_fmt << 10) | ((n >> 3) << 17) | (1u << 23) |
         ((128u >> 4) << 24) | (a_sf_id << 29);
}

// 32 lanes x 32-bit, 16 consecutive columns: thread i of the warp receives
// lane (quarter*32 + i), columns [col, col+16).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace moe
