// Device-side building blocks for sm_103a: mbarriers with bounded waits, bulk / tensor TMA
// copies, and the tcgen05 tensor-core instructions (TMEM allocation, MMA, commit, loads,
// shared-memory -> TMEM copies). Everything is inline PTX written against the PTX ISA
// (tcgen05 family, PTX 8.6+); no library code is used.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace hm {

// ------------------------------------------------------------------ device error word bits
constexpr uint32_t kErrHeader = 1u;    // packed header does not match the call
constexpr uint32_t kErrTimeout = 2u;   // a pipeline wait exceeded its time limit
constexpr uint32_t kErrOffsets = 4u;   // MoE offsets not monotone / out of range

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Diagnostics: record the global timer in slot `i` of this CTA's trace row (no-op when the
// caller installed no trace buffer).
__device__ __forceinline__ void trace_mark(uint64_t* trace, int i) {
  if (trace != nullptr) trace[blockIdx.x * 16 + i] = globaltimer();
}

// Diagnostics: per-stage / per-block stamps of CTA 0 (row r in 0..7, index i < 64) after the
// per-CTA rows.
__device__ __forceinline__ void trace_stage(uint64_t* trace, int r, int i) {
  if (trace != nullptr && blockIdx.x == 0 && i < 64) trace[256 * 16 + r * 64 + i] = globaltimer();
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Raise the expected transaction count of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\tmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same, but a thread whose phase has not completed is suspended until it completes or 20 us pass
// (the suspend-time hint) instead of returning at once, so that waiting warps leave the issue
// slots and the shared-memory pipe to the warps doing work. Measured 2-3 % faster on the
// 256-token W4A16 tiles (12 roles of 15 warps wait at any time) and 3-4 % slower on the
// bandwidth-bound decode kernels, which therefore poll.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\tmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2, 20000;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared state every role consults while waiting: a CTA-wide abort flag (set by the first
// role whose wait ran out, so the others stop instead of each waiting out its own limit),
// the global error word and the limit itself.
struct WaitCtx {
  volatile uint32_t* abort;  // shared memory
  uint32_t* err;             // global device error word
  uint64_t timeout_ns;
  bool suspend = false;      // wait with the suspend-time hint (mbar_try_wait_suspend)
};

// Waits until the barrier's phase with the given parity has completed. Returns false if the
// CTA is aborting or the wait exceeded ctx.timeout_ns (then sets kErrTimeout and the abort
// flag). Never spins without a limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& ctx) {
  const uint32_t a = smem_u32(bar);
  auto try_wait = [&]() { return ctx.suspend ? mbar_try_wait_suspend(a, parity) : mbar_try_wait(a, parity); };
  if (try_wait()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (try_wait()) return true;
    if (*ctx.abort) return false;
    if (globaltimer() - t0 > ctx.timeout_ns) {
      *ctx.abort = 1u;
      atomicOr(ctx.err, kErrTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------------------ thread-block clusters

// Split cluster barrier (per thread, not warp-aligned, so a warp may reach it from any branch).
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory object in the CTA of the cluster with the given rank.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Bounded wait for a phase completed by arrivals from other CTAs of the cluster (acquire at
// cluster scope, so their stores into this CTA's shared memory are visible afterwards).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, const WaitCtx& ctx) {
  const uint32_t a = smem_u32(bar);
  auto try_wait = [&]() {
    uint32_t ok;
    if (ctx.suspend)
      asm volatile(
          "{\n\t.reg .pred P;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2, 20000;\n\t"
          "selp.u32 %0, 1, 0, P;\n\t}"
          : "=r"(ok)
          : "r"(a), "r"(parity)
          : "memory");
    else
      asm volatile(
          "{\n\t.reg .pred P;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n\t"
          "selp.u32 %0, 1, 0, P;\n\t}"
          : "=r"(ok)
          : "r"(a), "r"(parity)
          : "memory");
    return ok != 0;
  };
  if (try_wait()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (try_wait()) return true;
    if (*ctx.abort) return false;
    if (globaltimer() - t0 > ctx.timeout_ns) {
      *ctx.abort = 1u;
      atomicOr(ctx.err, kErrTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------------------ async-proxy fences

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier for a subset of warps (id 1..15).
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ TMA

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0, both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 2-D tiled tensor copy global -> shared (x = innermost coordinate in elements).
__device__ __forceinline__ void tma_2d_g2s(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                           uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// CTA pairs: 2-D tiled copy into this CTA's shared memory whose completion is counted on a barrier
// of the pair's other CTA (`bar_cluster`: a shared::cluster address, from map_to_rank).
__device__ __forceinline__ void tma_2d_g2s_pair(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                uint32_t bar_cluster, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}

// 3-D tiled tensor copy global -> shared.
__device__ __forceinline__ void tma_3d_g2s(void* dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                           uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Programmatic dependent launch: let the next kernel in the stream start its prologue, and
// wait until every kernel this one depends on has finished and its writes are visible.
// Both are no-ops when the launch did not ask for programmatic serialization.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ tcgen05: TMEM management

// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); the TMEM address is
// written to *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// CTA pairs (a cluster of two CTAs whose tensor cores run one MMA together): the same
// allocation is made, and later freed, collectively by one warp of each CTA of the pair; every
// tcgen05 allocation, MMA and commit of such a kernel names the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05: descriptors

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle layout: rows of
// 128 bytes, 8-row atoms of 1024 bytes (stride between atoms = SBO = 1024), atom base
// 1024-byte aligned. Fields: start address >> 4 in bits 0-13, leading byte offset >> 4 in
// 16-29 (unused for swizzled K-major, set to 1), stride byte offset >> 4 in 32-45, the
// fixed value 0b001 in bits 46-48, base offset 0 in 49-51, swizzle mode in 61-63
// (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Descriptor of a scale-factor source for tcgen05.cp 32x128b: no swizzle, 8-row x 16-byte
// core matrices stacked contiguously (stride 128 bytes), LBO = 0.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 32) |
         (static_cast<uint64_t>(1) << 46);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9 = 1,
// 10-12 = 1), both K-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t m, uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Instruction descriptor for the block-scaled kinds (kind::mxf8f6f4, kind::mxf4nvf4):
// B scale-factor id in bits 4-5, A type in 7-9, B type in 10-12, N >> 3 in 17-22, scale
// type in bit 23 (1 = UE8M0, 0 = UE4M3), M >> 4 in 24-28, A scale-factor id in 29-30.
// Types for mxf8f6f4: e4m3 = 0, e2m1 = 5; for mxf4nvf4: e2m1 = 1.
__host__ __device__ constexpr uint32_t idesc_block_scaled(uint32_t m, uint32_t n, uint32_t atype,
                                                          uint32_t btype, uint32_t ue8m0,
                                                          uint32_t sfa_id, uint32_t sfb_id) {
  return (sfb_id << 4) | (atype << 7) | (btype << 10) | ((n >> 3) << 17) | (ue8m0 << 23) |
         ((m >> 4) << 24) | (sfa_id << 29);
}

// ------------------------------------------------------------------ tcgen05: MMA and friends

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same, with the A operand read from TMEM (M rows in lanes 0..M-1, two bf16 per 32-bit column
// along K; the 16 K of one instruction occupy 8 columns starting at a_tmem).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_mxf4nvf4_4x(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t sfa_tmem,
                                                uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05 async operations of this thread
// have completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// CTA-pair MMA, issued by one thread of the pair's even CTA: M = 256 rows of A, rows 0-127 from
// TMEM lanes 0-127 of the even CTA and rows 128-255 from the same TMEM address of the odd CTA; the
// N columns of B are split between the two CTAs' shared memory at the same address (the even CTA
// holds columns 0 .. N/2-1); each CTA's TMEM receives its 128 rows of D, all N columns.
__device__ __forceinline__ void mma_bf16_ta_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair version of tc_commit: arrive once on the barrier at the same shared-memory address in both
// CTAs of the pair when all previously issued tcgen05 operations of this thread have completed.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// Copy a 32-row x 128-bit block from shared memory into TMEM lanes 0-31 of 4 columns and
// replicate it into the other three 32-lane groups.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Whole warp: load 16 consecutive 32-bit columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Whole warp: load 16 TMEM lanes (from the lane in taddr, 16-aligned inside this warp's 32-lane
// group) x 32 consecutive 32-bit columns, in the layout of the warp-level MMA's accumulator
// fragment: for each group i of 8 columns, thread t receives in r[4i], r[4i+1] lane t/4, columns
// 8i + 2(t%4) and 8i + 2(t%4) + 1, and in r[4i+2], r[4i+3] lane t/4 + 8, the same two columns.
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Whole warp: store four 8x8 16-bit matrices to shared memory transposed. Register j of thread t
// holds elements (row t/4, columns 2(t%4) and 2(t%4) + 1) of matrix j (the lower column in the low
// half); the 16-byte shared address given by thread 8j + c receives column c of matrix j (its
// rows 0..7 in order).
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t saddr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(r0),
               "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

// Whole warp: store 32 consecutive 32-bit columns into this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ small helpers

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ __nv_bfloat162 bits_bf16x2(uint32_t v) {
  return *reinterpret_cast<__nv_bfloat162*>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

}  // namespace hm
