// W4A16 GEMM on tcgen05: Y[M,N] = X[M,K] * dequant(W)^T with 4-bit weights restored to bf16
// in registers and multiplied on the 5th-generation tensor cores (kind::f16, fp32 accumulate
// in TMEM). Dense and grouped-MoE variants.
//
// The computation is the explainer page's linear layer ("vLLM Humming은 4비트를 어떻게
// 계산하나", section "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다": Y = X * W^T, W
// stored [N,K], read once and reused over the M rows) with W replaced by its restored value
// (section "4비트 값에는 스케일이라는 해석 규칙이 붙는다"); the MoE variant is the same
// product per expert over that expert's contiguous token rows (MoE paragraph of the first
// section).
//
// Design (GB300-first; the pages give no kernel design):
//  * weights are the MMA's A operand (M = 128 weight rows), tokens its B operand (N =
//    tile_m in 16..256), so even M = 1 fills the 128-row side of the tensor core;
//  * one persistent CTA per SM, 15 warps: warp 0 issues the TMA loads (one bulk copy of g
//    contiguous packed 128x128 units with their scales, and the matching X tile), warps 1-2
//    issue tcgen05.mma (two issuers with separate accumulators for tile_m <= 64, warp 1 also
//    owns TMEM), warps 3-10 restore the weights to bf16 (two groups taking alternate 128-K
//    blocks) into TMEM (tile_m <= 128, the MMA reads A from TMEM) or into the 128-byte-swizzled
//    K-major shared layout (tile_m = 256), warps 11-14 drain TMEM (tcgen05.ld), round to bf16
//    and store Y;
//  * INT4 with tile_m 16 or 32 runs the small-token kernel instead (hm_gemm_f16s.cu);
//  * accumulators are double-buffered in TMEM so the epilogue of one tile overlaps the main
//    loop of the next;
//  * small M uses stream-K (hm_sched.cuh) so that every SM streams weights; the CTA holding a
//    tile's first k-block sums the other CTAs' published partials in k order (deterministic;
//    no contributor waits);
//  * programmatic dependent launch: the first weight stages stream before the wait for the
//    previous kernel; every wait is bounded (hm_device.cuh).
//
// This header holds the kernel template; hm_gemm_f16.cu (INT4 and the dispatch),
// hm_gemm_f16_mxfp4.cu and hm_gemm_f16_mxint4.cu instantiate it, one weight format each.
#pragma once
#include <cuda_bf16.h>

#include <cstdlib>

#include "hm_dequant.cuh"
#include "hm_device.cuh"
#include "hm_f16_common.cuh"
#include "hm_kernels.h"
#include "hm_layout.h"
#include "hm_sched.cuh"

namespace hm {
namespace {

// Dequant warps: two groups of four that take alternate 128-K blocks, so that two blocks are
// being restored at any time (one block's chain of shared loads, conversion, TMEM store and
// barrier signalling is latency-bound); inside a group each warp owns one 32-row TMEM quarter
// and each thread restores its row's whole 128-K block.
constexpr int kDqGroup = 4;
constexpr int kDqWarps = 2 * kDqGroup;
// Warp roles: 0 producer, 1-2 MMA issuers (warp 1 also owns TMEM), 3-10 dequant, 11-14 epilogue.
constexpr int kMmaWarp0 = 1;
constexpr int kDqWarp0 = 3;
constexpr int kEpiWarp0 = kDqWarp0 + kDqWarps;
constexpr int kThreads = 32 * (kEpiWarp0 + 4);
constexpr int kAStage = 128 * 128 * 2;  // restored bf16 weight tile, 2 swizzle atoms of 64 K

// Variants of the A (restored weight) path:
//  * tile_m <= 192: the dequant warps store bf16 A straight into TMEM (tcgen05.st) and the MMA
//    reads A from TMEM, so shared memory carries only the packed weights and X; TMEM holds the
//    double-buffered accumulator (2 x tile_m columns) plus kSA A stages of 64 columns (two at 192
//    tokens, whose accumulator pair takes 384 of the 512 columns);
//  * tile_m = 256 (T1 = false): the accumulator pair fills TMEM, so A goes through shared memory
//    in the 128-byte-swizzled K-major layout (two A stages);
//  * tile_m = 256, T1 = true: A in TMEM with four A stages beside a single accumulator; load
//    stages gain the shared memory A left (three instead of two). Each 128-K block then waits less
//    for its activations and restored weights (measured timelines: ~0.77 instead of ~1.0 us per
//    block), but the next tile's first MMA waits for the epilogue, so the planner takes it for long
//    K loops or few tiles per CTA.
//  * PAIR (dense): A in TMEM, and a cluster of two CTAs runs each MMA together (M = 256 weight
//    rows, 128 restored in each CTA's TMEM; N = tile_m tokens, half of the activation tile in each
//    CTA's shared memory), so a CTA loads half the activation bytes per weight row; tile_m 128 (two
//    accumulators) or 256 (one).
// A load stage holds kG consecutive 128-K blocks (one bulk copy of kG contiguous units and one
// activation load), so that small token tiles move many bytes per TMA instruction; the dequant
// warps and the MMA still step through it one 128-K block (one TMEM A slot) at a time.
// One thread issuing tcgen05.mma waits about 46 cycles per instruction whatever N, while the
// tensor core accepts M = 128 / K = 16 MMAs with A in TMEM several times faster from several
// threads. Small token tiles (N <= 64, where one MMA is far below that wait) therefore use two
// issuing warps that take alternate 128-K blocks into separate accumulators, which the epilogue
// adds (issuer 0 first, so the sum is deterministic).
template <int BT, int UB = kUnitMx, bool T1 = false, bool PAIR = false>
struct F16Shape {
  static constexpr bool kATmem = BT <= 192 || T1 || PAIR;
  static constexpr int kIss = BT <= 64 ? 2 : 1;
  // Accumulator buffers: two (the epilogue of one tile overlaps the next tile's main loop), or one
  // (T1, and pairs at 256 tokens: TMEM room for four A stages at 256 tokens).
  static constexpr int kAccBufs = (T1 || (PAIR && BT == 256)) ? 1 : 2;
  static constexpr int kAccCols = kAccBufs * kIss * BT;  // accumulator (issuer i, buffer b) at (b*kIss + i)*BT
  static constexpr int kXRows = PAIR ? BT / 2 : BT;      // activation rows (tokens) in this CTA's stages
  static constexpr int kG = f16_group_of(BT);
  static constexpr int kXStage = kG * kXRows * 128 * 2;
  static constexpr int kWStage = kG * UB;  // room for the largest units of the formats served
  static constexpr int kSA = kATmem ? ((512 - kAccCols) / 64 > 6 ? 6 : (512 - kAccCols) / 64) : 2;
  static constexpr int kAOff = 0;
  static constexpr int kASmem = kATmem ? 0 : kSA * kAStage;
  static constexpr int kXOff = kASmem;
  // One 128-K block per stage and a single issuer (tile_m >= 128): one commit per block signals
  // both the block's A slot and its load stage free (mma_done ring of kSD barriers); the issuing
  // thread spends about as long on a commit as on an MMA, so this saves an eighth of its work per
  // block. Otherwise each stage and each A slot has its own release barrier.
  static constexpr bool kMerged = kG == 1 && kIss == 1;
  // load stages: as many as shared memory holds beside the A stages, the barriers (at most 4 per
  // load stage and 2 per A slot), the MoE arrays of up to 1024 experts and the alignment slack
  // (smem_bytes(1024))
  static constexpr int kSLFit = (232448 - 1024 - kASmem - (2 * kSA + 5) * 8 - 96 - 8 * 1025) / (kXStage + kWStage + 32);
  static constexpr int kSL = kSLFit > 16 ? 16 : kSLFit;
  static constexpr int kSD = kMerged ? (kSA > kSL ? kSA : kSL) : kSA;   // MMA release barriers
  static constexpr int kWOff = kXOff + kSL * kXStage;
  static constexpr int kBarOff = kWOff + kSL * kWStage;
  // full_w, full_x, empty_l [kSL]; full_a [kSA]; empty_a / mma_done [kSD]; acc_full, acc_empty [2]; drain
  static constexpr int kNumBars = 3 * kSL + kSA + kSD + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kLutOff = kMiscOff + 32;
  static constexpr int kMoeOff = kLutOff + 64;
  static constexpr uint32_t kTmemCols = kATmem ? 512u : (2 * BT < 32 ? 32u : 2u * BT);
  static constexpr uint32_t kACol0 = kAccCols;  // first TMEM column of the A stages
  // MoE: offsets and tile prefix (8 (E + 1) bytes) at kMoeOff; then, where shared memory has room,
  // the epilogue warps' transpose scratch ([warp][16 tokens][32 rows] bf16), 16-byte aligned for its
  // vector loads
  static constexpr int kEpiScratch = 4 * 16 * 32 * 2;   // one 16-token chunk per warp (x2: two chunks)
  static constexpr __host__ __device__ int epi_off(int experts) {
    return (kMoeOff + (experts > 0 ? 8 * (experts + 1) : 0) + 15) / 16 * 16;
  }
  static constexpr int smem_bytes(int experts, int scratch_chunks = 0) {
    return 1024 + (scratch_chunks > 0 ? epi_off(experts) + scratch_chunks * kEpiScratch
                                      : kMoeOff + (experts > 0 ? 8 * (experts + 1) : 0));
  }
  static_assert(kSL >= 2, "load pipeline depth");
  static_assert(!PAIR || ((BT == 128 || BT == 256) && kMerged), "CTA pairs: 128 or 256 tokens");
  static_assert(smem_bytes(1024) <= 232448, "shared memory per CTA");
  static_assert(!kATmem || kACol0 + kSA * 64 <= 512, "TMEM budget");
  static_assert(kATmem || kIss == 1, "two issuers only with A in TMEM");
};

// Unit bytes a load stage must hold per 128-K block for a weight format (WK).
constexpr int f16_unit_room(int wk) {
  return wk == 8 ? static_cast<int>(kUnitInt8Zp) : (wk == 6 ? static_cast<int>(kUnitG32Zp) : static_cast<int>(kUnitMx));
}

// WK: 0 = INT4 (zero-points read from the packed header at run time), 2 = MXFP4, 3 = MXINT4,
// 6 = INT4 with a bf16 scale and u4 zero-point per 32-K chunk, 8 = INT8 (tiles up to 192 tokens).
template <int BT, int WK, bool MOE, bool T1, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) f16_gemm_kernel(const __grid_constant__ F16Params p) {
  using S = F16Shape<BT, f16_unit_room(WK), T1, PAIR>;
  static_assert(!(PAIR && MOE), "CTA pairs serve the dense product");
  constexpr int SL = S::kSL;
  constexpr int SA = S::kSA;
  constexpr int SD = S::kSD;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* full_w = bars;
  uint64_t* full_x = bars + SL;
  uint64_t* empty_l = bars + 2 * SL;
  uint64_t* full_a = bars + 3 * SL;
  uint64_t* empty_a = full_a + SA;   // merged releases: mma_done[SD], block bi completes on bi % SD
  uint64_t* acc_full = empty_a + SD;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + S::kMiscOff + 4);
  float* lut = reinterpret_cast<float*>(smem + S::kLutOff);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + S::kMoeOff);
  int32_t* offs = prefix + (MOE ? p.num_experts + 1 : 0);
  volatile uint32_t* hz_sh = reinterpret_cast<volatile uint32_t*>(smem + S::kMiscOff + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pairs: rank 0 issues the pair's MMAs; the other CTA's arrivals on its barriers are remote
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0u;

  if (MOE) {
    // The MoE prefix warp may raise the abort flag while thread 0 is still setting up: clear the
    // flag before any role runs, so that a raised flag is never overwritten.
    if (threadIdx.x == 0) *abort_flag = 0u;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    trace_mark(p.trace, 0);
    // Read the (first) weight header before initialising the barriers so that its memory
    // latency overlaps the set-up. MoE offsets (and thus expert pointers) may come from the
    // previous kernel, so the MoE variant waits for it first.
    if (MOE) pdl_wait();
    const uint8_t* first = (MOE && p.packed_list != nullptr) ? p.packed_list[0] : p.packed;
    const PackedHeader hdr = *reinterpret_cast<const PackedHeader*>(first);
    // Pairs: both CTAs' activation copies of a stage complete on the even CTA's full_x (the odd
    // CTA's stays unused); the even CTA's A slots and accumulators count both CTAs' warps.
    for (int s = 0; s < SL; ++s) {
      mbar_init(&full_w[s], 1);
      mbar_init(&full_x[s], 1);
      mbar_init(&empty_l[s], (S::kMerged ? 0 : S::kIss) + kDqWarps);
    }
    for (int s = 0; s < SA; ++s) mbar_init(&full_a[s], kDqGroup * (PAIR ? 2 : 1));
    for (int s = 0; s < SD; ++s) mbar_init(&empty_a[s], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], S::kIss);
      mbar_init(&acc_empty[b], 4 * (PAIR ? 2 : 1));
    }
    mbar_init(drain, S::kIss);
    fence_barrier_init();
    if (!MOE) *abort_flag = 0u;
    // The first weight's header decides whether INT4 units carry zero-points; every weight
    // used must agree with it and with the call's (fmt, N, K).
    const uint32_t hz = hdr.has_zero;
    *hz_sh = ((WK == 0 || WK == 6 || WK == 8) && hz == 1u) ? 1u : 0u;
    if (!(hdr.magic == kMagic && static_cast<int32_t>(hdr.fmt) == p.fmt && hdr.n == p.n && hdr.k == p.k)) {
      atomicOr(p.err, kErrHeader);
      *abort_flag = 1u;
    }
  }
  if (threadIdx.x < 16) lut[threadIdx.x] = e2m1_value(threadIdx.x);
  if (warp == kMmaWarp0) {
    if constexpr (PAIR) tmem_alloc_pair(tmem_slot, S::kTmemCols);
    else tmem_alloc(tmem_slot, S::kTmemCols);
  }
  if (MOE && warp == kDqWarp0) pdl_wait();   // the offsets below may be written by the previous kernel

  int32_t num_tiles = p.sched.num_tiles;
  if (MOE) {
    // Per-expert tile counts and their exclusive prefix (first dequant warp), offsets copied to shared.
    if (warp == kDqWarp0) moe_tile_prefix<BT>(p, offs, prefix, abort_flag, lane);
  }
  __syncthreads();
  if (PAIR) {   // both CTAs' barriers are initialised before either signals the other's
    cluster_arrive();
    cluster_wait();
  }
  tc_fence_after();
  if (MOE) num_tiles = prefix[p.num_experts];
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns, true};   // waiting roles suspend (mbar_try_wait_suspend)
  SchedIter sched;
  sched.init(p.sched, num_tiles, PAIR ? static_cast<int32_t>(blockIdx.x >> 1) : static_cast<int32_t>(blockIdx.x));
  const int kb_total = p.sched.kb_total;
  const bool aborted_early = *abort_flag != 0u;
  const uint32_t has_zero = *hz_sh;
  if (threadIdx.x == 0) {
    trace_mark(p.trace, 1);
    pdl_launch_dependents();
  }
  const uint32_t kUnit = WK == 8 ? (has_zero ? kUnitInt8Zp : kUnitInt8)
                         : WK == 6 ? (has_zero ? kUnitG32Zp : kUnitG32)
                                   : (WK >= 2 ? kUnitMx : (has_zero ? kUnitInt4Zp : kUnitInt4));
  // Weights are streamed once when a single token tile covers M; with several token tiles the
  // same weight tiles are read again by other CTAs, so keep them in L2.
  const bool reuse_w = MOE || p.num_m_tiles > 1;
  // Tile -> rows and weights. A pair's tile covers 256 weight rows (128 in each CTA) and BT tokens,
  // of which each CTA loads the activations of BT / 2.
  auto tile_info = [&](int tile) -> TileInfo {
    if constexpr (PAIR) {
      const int np = p.num_n_tiles >> 1;
      const int nt = 2 * (tile % np) + static_cast<int>(rank);
      TileInfo t;
      t.m0 = (tile / np) * BT;
      t.m_end = static_cast<int32_t>(p.m < t.m0 + BT ? p.m : t.m0 + BT);
      t.n0 = nt * 128;
      t.base = p.packed;
      t.wbase = p.packed + kHeaderBytes + static_cast<size_t>(nt) * kb_total * kUnit;
      return t;
    } else {
      return decode_tile<BT, MOE>(p, tile, prefix, offs, kUnit);
    }
  };
  const int x_row0 = PAIR ? static_cast<int>(rank) * (BT / 2) : 0;   // this CTA's first token in a tile

  if (aborted_early) {
    // nothing to do: fall through to teardown
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tmap_x);
      const uint64_t pol_w = reuse_w ? policy_evict_last() : policy_evict_first();
      const uint64_t pol_x = reuse_w ? policy_evict_normal() : policy_evict_last();
      const uint8_t* last_checked = nullptr;
      // A weight buffer is read only after its header matched the call (MoE: each expert's).
      auto checked = [&](const TileInfo& t) -> bool {
        if (!MOE || t.base == last_checked) return true;
        if (!header_ok(t.base, p, has_zero)) {
          atomicOr(p.err, kErrHeader);
          *abort_flag = 1u;
          return false;
        }
        last_checked = t.base;
        return true;
      };
      // Stage `idx` (ring slot idx % SL) covers k-blocks [kb, kb + g) of tile t.
      auto issue_w = [&](int idx, const TileInfo& t, int kb, int g) {
        const int slot = idx % SL;
        const uint32_t bytes = static_cast<uint32_t>(g) * kUnit;
        mbar_arrive_expect_tx(&full_w[slot], bytes);
        bulk_g2s(smem + S::kWOff + slot * S::kWStage, t.wbase + static_cast<size_t>(kb) * kUnit, bytes,
                 &full_w[slot], pol_w);
      };
      auto issue_x = [&](int idx, const TileInfo& t, int kb) {
        const int slot = idx % SL;
        uint8_t* xs = smem + S::kXOff + slot * S::kXStage;
        trace_stage(p.trace, 0, idx);
        if constexpr (PAIR) {
          // the even CTA expects both halves; the odd CTA's copies complete on the even CTA's barrier
          if (!leader) {
            const uint32_t bar = map_to_rank(smem_u32(&full_x[slot]), 0);
            tma_2d_g2s_pair(xs, &p.tmap_x, kb * 128, t.m0 + x_row0, bar, pol_x);
            tma_2d_g2s_pair(xs + S::kXRows * 128, &p.tmap_x, kb * 128 + 64, t.m0 + x_row0, bar, pol_x);
          } else {
            mbar_arrive_expect_tx(&full_x[slot], 2 * S::kXStage);
            tma_2d_g2s(xs, &p.tmap_x, kb * 128, t.m0, &full_x[slot], pol_x);
            tma_2d_g2s(xs + S::kXRows * 128, &p.tmap_x, kb * 128 + 64, t.m0, &full_x[slot], pol_x);
          }
        } else if constexpr (S::kG == 1) {
          mbar_arrive_expect_tx(&full_x[slot], S::kXStage);   // the whole box lands (zero-filled past K)
          tma_2d_g2s(xs, &p.tmap_x, kb * 128, t.m0, &full_x[slot], pol_x);
          tma_2d_g2s(xs + BT * 128, &p.tmap_x, kb * 128 + 64, t.m0, &full_x[slot], pol_x);
        } else {
          mbar_arrive_expect_tx(&full_x[slot], S::kXStage);
          tma_3d_g2s(xs, &p.tmap_x, 0, t.m0, 2 * kb, &full_x[slot], pol_x);
        }
        if (idx == 0) trace_mark(p.trace, 2);
      };
      // Start-up order. The weights of stage 0 do not depend on the previous kernel, so the
      // dense path streams them before waiting for it. Then the activation tiles of the first SL
      // stages go out before the rest of their weights: an SM's copies complete roughly in issue
      // order, and an activation tile queued behind ~100 KB of weights would hold back the first
      // MMA by microseconds.
      int issued_w = 0, issued_x = 0;
      bool ok = true;
      if (!MOE) {
        SchedIter pf = sched;
        Segment ps;
        if (pf.next(ps)) {
          const TileInfo t = tile_info(ps.tile);
          issue_w(0, t, ps.kb0, min(S::kG, ps.kb1 - ps.kb0));
          issued_w = 1;
        }
      }
      pdl_wait();
      {
        SchedIter pf = sched;
        Segment ps;
        int idx = 0;
        while (idx < SL && pf.next(ps)) {
          const TileInfo t = tile_info(ps.tile);
          for (int kb = ps.kb0; kb < ps.kb1 && idx < SL; kb += S::kG, ++idx) issue_x(idx, t, kb);
        }
        issued_x = idx;
        pf = sched;
        idx = 0;
        while (idx < issued_x && pf.next(ps)) {
          const TileInfo t = tile_info(ps.tile);
          if (!checked(t)) { ok = false; break; }
          for (int kb = ps.kb0; kb < ps.kb1 && idx < issued_x; kb += S::kG, ++idx)
            if (idx >= issued_w) issue_w(idx, t, kb, min(S::kG, ps.kb1 - kb));
        }
        if (ok) issued_w = issued_x;
      }
      // Steady state: a stage is refilled once every consumer released it (merged releases: the
      // dequant warps on empty_l, the MMAs of the stage's block on its mma_done barrier).
      int idx = 0;
      int ls = 0;
      uint32_t lph = 0;
      Segment seg;
      while (ok && sched.next(seg)) {
        const TileInfo t = tile_info(seg.tile);
        if (!checked(t)) break;
        for (int kb = seg.kb0; kb < seg.kb1; kb += S::kG, ++idx) {
          if (idx >= issued_x) {
            if (!mbar_wait(&empty_l[ls], lph ^ 1u, wc)) { ok = false; break; }
            if (S::kMerged) {
              const int j = idx - SL;   // the block that last used this stage
              if (!mbar_wait(&empty_a[j % SD], static_cast<uint32_t>(j / SD) & 1u, wc)) { ok = false; break; }
            }
            issue_w(idx, t, kb, min(S::kG, seg.kb1 - kb));   // weights first: the dequant needs them first
            issue_x(idx, t, kb);
            issued_x = issued_w = idx + 1;
          }
          if (++ls == SL) { ls = 0; lph ^= 1u; }
        }
      }
      trace_mark(p.trace, 3);
      if (*abort_flag) {
        // Let copies already in flight (at most the last SL stages issued) land before the
        // CTA's shared memory goes away. A pair's activation copies complete on the even CTA's
        // barriers, whose phases also need the other CTA's copies, so pairs wait a fixed 200 us
        // for them instead (at most SL stages from L2 or HBM land within microseconds).
        if (PAIR) {
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 200000ull) {
          }
        } else {
          for (int i = issued_x > SL ? issued_x - SL : 0; i < issued_x; ++i)
            drain_wait(&full_x[i % SL], static_cast<uint32_t>(i / SL) & 1u, 100000000ull);
        }
        for (int i = issued_w > SL ? issued_w - SL : 0; i < issued_w; ++i)
          drain_wait(&full_w[i % SL], static_cast<uint32_t>(i / SL) & 1u, 100000000ull);
      }
    }
  } else if (warp < kMmaWarp0 + S::kIss) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer `is` takes the 128-K blocks whose running sequence index bi has bi % kIss == is,
    // accumulating into its own TMEM accumulator; A slot bi % SA holds block bi.
    // Pairs: the even CTA issues for both; barriers the odd CTA also arrives on (or whose copies
    // complete there) are waited at cluster scope, and every commit signals both CTAs.
    if (lane == 0 && leader) {
      const int is = warp - kMmaWarp0;
      constexpr uint32_t idesc = idesc_bf16(PAIR ? 256 : 128, BT);
      auto wait_c = [&](uint64_t* bar, uint32_t parity) -> bool {
        if constexpr (PAIR) return mbar_wait_cluster(bar, parity, wc);
        else return mbar_wait(bar, parity, wc);
      };
      auto commit = [&](uint64_t* bar) {
        if constexpr (PAIR) tc_commit_pair(bar);
        else tc_commit(bar);
      };
      int ls = 0;
      uint32_t lph = 0, acc_i = 0;
      int seq = 0;
      Segment seg;
      bool ok = true;
      while (ok && sched.next(seg)) {
        const uint32_t b = acc_i % S::kAccBufs;
        if (!wait_c(&acc_empty[b], ((acc_i / S::kAccBufs) & 1u) ^ 1u)) break;
        tc_fence_after();
        const uint32_t d = tmem + (b * S::kIss + is) * BT;
        bool first = true;
        for (int kb0 = seg.kb0; kb0 < seg.kb1 && ok; kb0 += S::kG) {
          // Wait for the stage even without a block in it: the release below must not reach
          // the slot's empty barrier before the slot's previous use is over. (Merged releases: the
          // dequant warps saw the activations land before they marked the block's A slot full.)
          if (!S::kMerged && !wait_c(&full_x[ls], lph)) { ok = false; break; }
          if (is == 0) trace_stage(p.trace, 7, seq / S::kG);
          const int g = min(S::kG, seg.kb1 - kb0);
          for (int j = 0; j < g; ++j) {
            const int bi = seq + j;
            if (S::kIss > 1 && bi % S::kIss != is) continue;
            const int as = bi % SA;
            const uint32_t aph = static_cast<uint32_t>(bi / SA) & 1u;
            if (!wait_c(&full_a[as], aph)) { ok = false; break; }
            trace_stage(p.trace, 3, bi);
            tc_fence_after();
            if (is == 0 && acc_i == 0 && first) trace_mark(p.trace, 6);
            trace_stage(p.trace, 4, bi);
            const uint32_t x_base = smem_u32(smem + S::kXOff + ls * S::kXStage) + j * (2 * S::kXRows * 128);
            if constexpr (PAIR) {
              const uint32_t a_t = tmem + S::kACol0 + as * 64;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint64_t bd = sdesc_sw128(x_base + (k >> 2) * (S::kXRows * 128) + (k & 3) * 32);
                mma_bf16_ta_pair(d, a_t + 8 * k, bd, idesc, (!first || k > 0) ? 1u : 0u);
              }
            } else if constexpr (S::kATmem) {
              const uint32_t a_t = tmem + S::kACol0 + as * 64;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint64_t bd = sdesc_sw128(x_base + (k >> 2) * (BT * 128) + (k & 3) * 32);
                mma_bf16_ta(d, a_t + 8 * k, bd, idesc, (!first || k > 0) ? 1u : 0u);
              }
            } else {
              const uint32_t a_base = smem_u32(smem + S::kAOff + as * kAStage);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint64_t ad = sdesc_sw128(a_base + (k >> 2) * (kAStage / 2) + (k & 3) * 32);
                const uint64_t bd = sdesc_sw128(x_base + (k >> 2) * (BT * 128) + (k & 3) * 32);
                mma_bf16(d, ad, bd, idesc, (!first || k > 0) ? 1u : 0u);
              }
            }
            first = false;
            trace_stage(p.trace, 5, bi);
            if (S::kMerged) commit(&empty_a[bi % SD]);   // the block's A slot and load stage
            else commit(&empty_a[as]);
            trace_stage(p.trace, 6, bi);
          }
          if (!ok) break;
          if (!S::kMerged) commit(&empty_l[ls]);
          seq += g;
          if (++ls == SL) { ls = 0; lph ^= 1u; }
        }
        if (!ok) break;
        commit(&acc_full[b]);   // also when this issuer had no block in the tile
        ++acc_i;
      }
      if (is == 0) trace_mark(p.trace, 7);
      // All tcgen05 work of this thread has completed once `drain` flips (one arrival per issuer).
      commit(drain);
      drain_wait(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= kDqWarp0 && warp < kEpiWarp0) {
    // ------------------------------------------------------------ dequant warps
    // Warp -> (group, row, K half). With A in TMEM a warp may only touch its own 32-lane
    // quarter (warp index % 4), so rows follow the quarter; otherwise rows follow the thread.
    const int dw = warp - kDqWarp0;
    const int grp = dw / kDqGroup;                 // takes the blocks with sequence index % 2 == grp
    const int r = 32 * (warp & 3) + lane;          // weight row within the tile (TMEM lane)
    int ls = 0;
    uint32_t lph = 0;
    int seq = 0;                                   // running 128-K block index over all segments
    bool first_dq = true;
    Segment seg;
    bool ok = true;
    while (ok && sched.next(seg)) {
      for (int kb0 = seg.kb0; kb0 < seg.kb1 && ok; kb0 += S::kG) {
        const int g = min(S::kG, seg.kb1 - kb0);
        // blocks j of this stage that belong to this group
        const int j0 = ((seq & 1) == grp) ? 0 : 1;
        // Every group waits for the stage to fill, even one with no block in it: its release
        // must not reach the ring slot's empty barrier before the slot's previous use is over,
        // or it would count towards the wrong phase.
        if (!mbar_wait(&full_w[ls], lph, wc)) {
          ok = false;
          break;
        }
        if (j0 >= g) {                             // none of the blocks: release the stage
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_l[ls]);
        }
        for (int jb = j0; jb < g; jb += 2) {
        const int bi = seq + jb;
        const int as = bi % SA;
        const uint32_t aph = static_cast<uint32_t>(bi / SA) & 1u;
        if (S::kMerged) {   // A slot free once the MMAs of block bi - SA completed
          const int jd = bi - SA;
          if (jd >= 0 && !mbar_wait(&empty_a[jd % SD], static_cast<uint32_t>(jd / SD) & 1u, wc)) { ok = false; break; }
        } else if (!mbar_wait(&empty_a[as], aph ^ 1u, wc)) {
          ok = false;
          break;
        }
        if (dw == 0 && first_dq) { trace_mark(p.trace, 4); first_dq = false; }
        if (dw % kDqGroup == 0 && lane == 0) trace_stage(p.trace, 1, bi);
        const uint32_t wsa = smem_u32(smem + S::kWOff + ls * S::kWStage) + jb * kUnit;
        if constexpr (WK != 8) {
          // INT4 and MXINT4 take the whole 128-K row into registers at once; MXFP4 (whose scale
          // and conversion need more registers) takes the second half after converting the first.
          uint4 c[4];
  #pragma unroll
          for (int i = 0; i < (WK == 2 ? 2 : 4); ++i) c[i] = ld_shared_v4(wsa + i * 2048 + r * 16);
          __nv_bfloat162 zz, ss;
          uint32_t e4 = 0;
          uint32_t s4[2] = {0u, 0u}, z4 = 0x8888u;   // WK 6: the four chunks' bf16 scales and zero-points
          if (WK == 6) {
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(s4[0]), "=r"(s4[1]) : "r"(wsa + kUnitCodes + 8 * r));
            if (has_zero) {
              uint16_t zb;
              asm volatile("ld.shared.u16 %0, [%1];" : "=h"(zb) : "r"(wsa + kUnitG32 + 2 * r));
              z4 = zb;
            }
            zz = int4_zero_pair(8);
            ss = bf16_pair(0);
          } else if (WK >= 2) {
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(e4) : "r"(wsa + kUnitCodes + 4 * r));
            zz = int4_zero_pair(8);   // MXINT4 nibbles are q + 8
          } else {
            uint16_t sb;
            asm volatile("ld.shared.b16 %0, [%1];" : "=h"(sb) : "r"(wsa + kUnitCodes + 2 * r));
            ss = bf16_pair(sb);
            uint32_t z = 8u;
            if (has_zero) {
              uint16_t zb;
              asm volatile("ld.shared.u8 %0, [%1];" : "=h"(zb) : "r"(wsa + kUnitInt4 + (r >> 1)));
              z = (static_cast<uint32_t>(zb) >> (4 * (r & 1))) & 0xFu;
            }
            zz = int4_zero_pair(z);
          }
          const bool last_of_stage = jb + 2 >= g;
          if (WK != 2 && last_of_stage) {   // the stage's last block of this group is in registers
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_l[ls]);
          }
  #pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (WK == 2 && half == 1) {
  #pragma unroll
              for (int i = 2; i < 4; ++i) c[i] = ld_shared_v4(wsa + i * 2048 + r * 16);
              if (last_of_stage) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_l[ls]);
              }
            }
            uint32_t a_regs[32];  // TMEM path: 64 restored K of this row as bf16x2, in K order
  #pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int c4 = 2 * half + i;
              const uint32_t words[4] = {c[c4].x, c[c4].y, c[c4].z, c[c4].w};
              const uint32_t ex = (e4 >> (8 * c4)) & 0xFFu;
              const bool mx_bits = WK == 2 && ex <= 128u;
              const uint32_t sc2 = mx_pow2_pair(ex);
              const float scale = WK == 2 ? pow2f(static_cast<int>(ex) - 127) : 0.f;
              const __nv_bfloat162 si = bits_bf16x2(mxint_scale_pair(ex));
  #pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t o[4];
                if (WK == 6)
                  dq_int4_word(words[j], int4_zero_pair((z4 >> (4 * c4)) & 0xFu),
                               bf16_pair(static_cast<uint16_t>(s4[c4 >> 1] >> (16 * (c4 & 1)))), o);
                else if (WK == 0) dq_int4_word(words[j], zz, ss, o);
                else if (WK == 3) dq_int4_word(words[j], zz, si, o);
                else if (mx_bits) dq_mx_word_bits(words[j], sc2, o);
                else dq_mx_word(words[j], lut, scale, o);
                if constexpr (S::kATmem) {
  #pragma unroll
                  for (int t = 0; t < 4; ++t) a_regs[16 * i + 4 * j + t] = o[t];
                } else {
                  const int ch = 4 * c4 + j;  // 16-byte chunk (8 consecutive K) within the 128 K
                  const uint32_t a_base = smem_u32(smem + S::kAOff + as * kAStage);
                  const uint32_t dst = a_base + (ch >> 3) * (kAStage / 2) + r * 128 +
                                       ((static_cast<uint32_t>(ch & 7) ^ static_cast<uint32_t>(r & 7)) << 4);
                  st_shared_v4(dst, o[0], o[1], o[2], o[3]);
                }
              }
            }
            if constexpr (S::kATmem)
              tmem_st32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + S::kACol0 + as * 64 + half * 32, a_regs);
          }
        } else {
          // INT8: one byte per code, the row's 128 codes in 8 chunks of 16; scale and zero-point per
          // row; the two 64-K halves are loaded, restored and stored to TMEM in turn
          static_assert(S::kATmem, "INT8 tiles keep the restored weights in TMEM");
          uint16_t sb;
          asm volatile("ld.shared.b16 %0, [%1];" : "=h"(sb) : "r"(wsa + kUnitInt8Codes + 2 * r));
          const __nv_bfloat162 s8 = bf16_pair(sb);
          uint32_t zb = 128u;
          if (has_zero) {
            uint16_t z16;
            asm volatile("ld.shared.u8 %0, [%1];" : "=h"(z16) : "r"(wsa + kUnitInt8 + r));
            zb = z16;
          }
          const float zf = 8388608.0f + static_cast<float>(zb);
          const bool last_of_stage = jb + 2 >= g;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint4 c8[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) c8[i] = ld_shared_v4(wsa + (4 * half + i) * 2048 + r * 16);
            if (half == 1 && last_of_stage) {   // the stage's last block of this group is in registers
              __syncwarp();
              if (lane == 0) mbar_arrive(&empty_l[ls]);
            }
            uint32_t a_regs[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t words[4] = {c8[i].x, c8[i].y, c8[i].z, c8[i].w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t p2[2];
                dq_int8_word(words[j], zf, s8, p2);
                a_regs[8 * i + 2 * j] = p2[0];
                a_regs[8 * i + 2 * j + 1] = p2[1];
              }
            }
            tmem_st32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + S::kACol0 + as * 64 + half * 32, a_regs);
          }
        }
        if constexpr (S::kATmem) {
          tmem_wait_st();
          tc_fence_before();
        } else {
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (dw % kDqGroup == 0 && lane == 0) trace_stage(p.trace, 2, bi);
        // Merged releases: the group's first warp also waits for the block's activations, so that
        // the MMA issuer waits on one barrier per block (pairs: the even CTA's, which counts both
        // halves).
        if (S::kMerged && dw % kDqGroup == 0 && leader && lane == 0) {
          const bool landed = PAIR ? mbar_wait_cluster(&full_x[ls], lph, wc) : mbar_wait(&full_x[ls], lph, wc);
          if (!landed) ok = false;
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          if (PAIR && !leader) mbar_arrive_remote(map_to_rank(smem_u32(&full_a[as]), 0));
          else mbar_arrive(&full_a[as]);
        }
        }
        seq += g;
        if (++ls == SL) { ls = 0; lph ^= 1u; }
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue warps (last four)
    pdl_wait();                          // Y, partials and counters may be in use by the previous kernel
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int row = 32 * q + lane;       // weight row within the tile
    // the flattened (tile, k-block) space of the stream-K tiles (all tiles, or the leading ones of
    // a hybrid schedule): the hand-off indexes CTAs' ranges in it
    const int64_t total_it = static_cast<int64_t>(sk_tiles_of(p.sched, num_tiles)) * kb_total;
    // 16-byte stores of Y through the transpose scratch (when the launch has one; Y 16-byte aligned,
    // N % 8 == 0)
    const bool vec_y = p.epi_scratch && (reinterpret_cast<uintptr_t>(p.y) & 15u) == 0 && (p.n & 7) == 0;
    // This warp's transpose scratch: [16 tokens][32 rows] bf16 per chunk (the second chunk, where the
    // launch has room for it, 4 KB further).
    const uint32_t sc = smem_u32(smem + S::epi_off(MOE ? p.num_experts : 0)) + static_cast<uint32_t>(q) * (16 * 32 * 2);
    // Transpose through shared memory so that each store moves 8 consecutive rows (16 bytes) of one
    // token instead of one bf16 per thread: put() writes a thread's 16 tokens of its row, out() then
    // has each lane store 8 rows of one token (after a __syncwarp between them).
    auto put = [&](const uint32_t (&v)[16], uint32_t buf) {
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const uint16_t hb = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[jj])));
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(buf + (jj * 32 + lane) * 2), "h"(hb) : "memory");
      }
    };
    // swz: the 16-byte group of rows 8 c8 .. + 7 of token tt sits at slot c8 ^ ((tt >> 1) & 3) of the
    // token's 64 bytes (the layout the transposing matrix stores write without bank conflicts)
    auto out = [&](uint32_t buf, const TileInfo& t, int j0, bool swz) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int piece = lane + 32 * h;   // token piece / 4, rows 8 (piece % 4) .. + 7
        const int tt = piece >> 2, c8 = piece & 3;
        const int slot = swz ? (c8 ^ ((tt >> 1) & 3)) : c8;
        const uint4 v8 = ld_shared_v4(buf + (tt * 32 + 8 * slot) * 2);
        const int64_t m = static_cast<int64_t>(t.m0) + j0 + tt;
        const int64_t n8 = static_cast<int64_t>(t.n0) + 32 * q + 8 * c8;
        if (m < t.m_end) {
          if (n8 + 8 <= p.n) {
            *reinterpret_cast<uint4*>(p.y + m * p.n + n8) = v8;
          } else {
            const uint32_t w4[4] = {v8.x, v8.y, v8.z, v8.w};
            for (int e = 0; e < 8 && n8 + e < p.n; ++e)
              p.y[m * p.n + n8 + e] = __ushort_as_bfloat16(static_cast<uint16_t>(w4[e >> 1] >> (16 * (e & 1))));
          }
        }
      }
    };
    // Rows' values of tokens j0 .. j0 + 15 of tile t to Y (bf16, RNE): 16-byte stores through the
    // scratch when the launch has it, else one bf16 per thread and token.
    auto store_y = [&](const float (&a)[16], const TileInfo& t, int j0, int64_t n) {
      if (vec_y) {
        uint32_t va[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) va[jj] = __float_as_uint(a[jj]);
        put(va, sc);
        __syncwarp();
        out(sc, t, j0, false);
        __syncwarp();   // the scratch is rewritten by the next chunk
      } else if (n < p.n) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int64_t m = static_cast<int64_t>(t.m0) + j0 + jj;
          if (m < t.m_end) p.y[m * p.n + n] = __float2bfloat16_rn(a[jj]);
        }
      }
    };
    uint32_t acc_i = 0;
    bool first_seg = true;
    int seq = 0;                         // running 128-K block index, as the issuers count it
    Segment seg;
    while (sched.next(seg)) {
      const uint32_t b = acc_i % S::kAccBufs;
      // Issuer i wrote its accumulator iff the segment has a block with sequence index % 2 == i.
      const int nb = seg.kb1 - seg.kb0;
      const bool use1 = S::kIss > 1 && (nb >= 2 || (seq & 1) == 1);
      const bool use0 = S::kIss == 1 || nb >= 2 || (seq & 1) == 0;
      seq += nb;
      if (!mbar_wait(&acc_full[b], (acc_i / S::kAccBufs) & 1u, wc)) break;
      tc_fence_after();
      if (row == 0 && acc_i == 0) trace_mark(p.trace, 8);
      const TileInfo t = tile_info(seg.tile);
      const int64_t n = static_cast<int64_t>(t.n0) + row;
      const bool full = seg.kb0 == 0 && seg.kb1 == kb_total;
      // Stream-K tile shared by CTAs c_lo .. c_hi: the owner (holding k-block 0) waits for the
      // others' published partials and adds them to its own accumulator; the others publish.
      // With a single accumulator (kAccBufs == 1) the owner defers that sum: it stores its own
      // partial like a publisher, frees the accumulator for the next tile's MMAs at once, and then
      // adds its partial and the others' in the same order (so the result is the same bits).
      const bool owner = !full && seg.kb0 == 0;
      const bool defer = S::kAccBufs == 1 && !MOE && !PAIR && owner;   // (only dense single CTAs split K)
      uint32_t* flag = full ? nullptr
                            : sk_flag(p.counters, owner ? blockIdx.x
                                                        : sk_tile_owner(seg.tile, kb_total, total_it, p.sched.grid), q);
      int64_t c_hi = 0;
      bool have = true;
      if (owner && !defer) {
        c_hi = sk_owner(static_cast<int64_t>(seg.tile + 1) * kb_total - 1, total_it, p.sched.grid);
        have = sk_wait(flag, static_cast<uint32_t>(c_hi - blockIdx.x), wc);
        if (row == 0) trace_mark(p.trace, 10);
      }
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + b * S::kIss * BT;
      float* slot = p.partial + (static_cast<size_t>(blockIdx.x) * 2 + (first_seg ? 0 : 1)) * BT * 128 +
                    static_cast<size_t>(row) * BT;
      // Whole tiles with one issuer and room for two chunks of scratch: 32 tokens at a time. The
      // accumulator is read in the warp-level MMA's fragment layout (two 16-lane halves) and each
      // group of 8 tokens goes to the scratch as four 8x8 matrices (this warp's rows 0-7, 8-15,
      // 16-23, 24-31) stored transposed: token m's 32 rows land in its 64 bytes of scratch, rows
      // 8j .. 8j + 7 at 16-byte slot j ^ ((m >> 1) & 3); the bf16 rounding is put()'s (RNE per
      // element).
      const bool two = S::kIss == 1 && full && vec_y && p.epi_scratch == 2;
#pragma unroll 1
      for (int j0 = 0; two && j0 < BT; j0 += 32) {
        uint32_t lo[16], hi[16];   // TMEM lanes 32q + 0..15 and 32q + 16..31, tokens j0 .. j0 + 31
        tmem_ld_16x256b_x4(tbase + j0, lo);
        tmem_ld_16x256b_x4(tbase + (16u << 16) + j0, hi);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // tokens j0 + 8i .. + 7: chunk i / 2, its tokens 8 (i % 2) ..
          auto pk = [](uint32_t a, uint32_t b) {
            return bf16x2_bits(__floats2bfloat162_rn(__uint_as_float(a), __uint_as_float(b)));
          };
          // lane 8j + c gives the address of token 8 (i % 2) + c, rows 8j .. 8j + 7; swizzled so that
          // the 8 addresses of each matrix fall in 8 different bank groups
          const int tok = 8 * (i & 1) + (lane & 7);
          const int slot = (lane >> 3) ^ ((tok >> 1) & 3);
          const uint32_t dst = sc + static_cast<uint32_t>(i >> 1) * S::kEpiScratch +
                               static_cast<uint32_t>((tok * 32 + 8 * slot) * 2);
          stmatrix_x4_trans(dst, pk(lo[4 * i], lo[4 * i + 1]), pk(lo[4 * i + 2], lo[4 * i + 3]),
                            pk(hi[4 * i], hi[4 * i + 1]), pk(hi[4 * i + 2], hi[4 * i + 3]));
        }
        __syncwarp();
        out(sc, t, j0, true);
        out(sc + S::kEpiScratch, t, j0 + 16, true);
        __syncwarp();   // the scratch is rewritten by the next pair of chunks
      }
#pragma unroll 1
      for (int j0 = 0; !two && j0 < BT && have; j0 += 16) {
        uint32_t v[16];
        tmem_ld16(tbase + (use0 ? 0 : BT) + j0, v);
        if (S::kIss > 1 && use0 && use1) {
          uint32_t v1[16];
          tmem_ld16(tbase + BT + j0, v1);
          tmem_wait_ld();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) v[jj] = __float_as_uint(__uint_as_float(v[jj]) + __uint_as_float(v1[jj]));
        } else {
          tmem_wait_ld();
        }
        if ((full || owner) && !defer) {
          float a[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) a[jj] = __uint_as_float(v[jj]);
          if (owner)
            sk_add_partials<BT>(p.partial, total_it, p.sched.grid, kb_total, seg.tile, blockIdx.x, c_hi, row, j0, a);
          store_y(a, t, j0, n);
        } else {
          float4* dst = reinterpret_cast<float4*>(slot + j0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && !leader) mbar_arrive_remote(map_to_rank(smem_u32(&acc_empty[b]), 0));
        else mbar_arrive(&acc_empty[b]);
      }
      ++acc_i;
      if (row == 0) trace_mark(p.trace, 9);
      if (defer) {   // this thread reads back only its own row of the partial it stored above
        c_hi = sk_owner(static_cast<int64_t>(seg.tile + 1) * kb_total - 1, total_it, p.sched.grid);
        have = sk_wait(flag, static_cast<uint32_t>(c_hi - blockIdx.x), wc);
        if (row == 0) trace_mark(p.trace, 10);
#pragma unroll 1
        for (int j0 = 0; j0 < BT && have; j0 += 16) {
          float a[16];
          const float4* own = reinterpret_cast<const float4*>(slot + j0);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 f = __ldcg(own + i);
            a[4 * i] = f.x;
            a[4 * i + 1] = f.y;
            a[4 * i + 2] = f.z;
            a[4 * i + 3] = f.w;
          }
          sk_add_partials<BT>(p.partial, total_it, p.sched.grid, kb_total, seg.tile, blockIdx.x, c_hi, row, j0, a);
          store_y(a, t, j0, n);
        }
      }
      if (!full && !owner) sk_publish(flag, lane);
      if (owner && have) {
        __syncwarp();
        if (lane == 0) *flag = 0u;
        if (row == 0) trace_mark(p.trace, 11);
      }
      first_seg = false;
    }
  }

  __syncwarp();  // reconverge lanes that skipped a single-thread role before the CTA barrier
  __syncthreads();
  if (PAIR) {   // neither CTA frees its TMEM or shared memory while the other may still reach them
    cluster_arrive();
    cluster_wait();
  }
  if (warp == kMmaWarp0) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, S::kTmemCols);
    else tmem_dealloc(tmem, S::kTmemCols);
    if (lane == 0) {
      trace_mark(p.trace, 12);
      if (p.trace) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        p.trace[blockIdx.x * 16 + 13] = smid;
      }
    }
  }
}

template <int BT, int WK, bool MOE, bool T1 = false, bool PAIR = false>
cudaError_t launch_one(const F16Params& p, cudaStream_t st) {
  using S = F16Shape<BT, f16_unit_room(WK), T1, PAIR>;
  auto kern = f16_gemm_kernel<BT, WK, MOE, T1, PAIR>;
  // with the epilogue's transpose scratch where it fits beside the MoE arrays
  const int experts = MOE ? p.num_experts : 0;
  // two chunks of scratch where they fit (the epilogue then transposes two 16-token chunks at once)
  const int scratch = S::smem_bytes(experts, 2) <= 232448 ? 2 : (S::smem_bytes(experts, 1) <= 232448 ? 1 : 0);
  const int smem = S::smem_bytes(experts, scratch);
  F16Params q = p;
  q.epi_scratch = scratch;
  // Raise the dynamic shared-memory limit once per device (to the largest size any call of this
  // instantiation can ask for), so that later calls, including ones under stream capture, only launch.
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  if constexpr (!PAIR) {
    return launch_pdl(kern, q.sched.grid, kThreads, smem, st, q);
  } else {
    // q.sched.grid counts pairs: clusters of two CTAs, no more than the device holds at once
    // (taken once per device; dense launches of one instantiation all ask for the same shared memory).
    static int max_pairs[64] = {};
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(static_cast<unsigned>(kThreads));
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    if (max_pairs[dev] == 0) {
      cfg.gridDim = dim3(2u * static_cast<unsigned>(q.sched.grid));
      cfg.dynamicSmemBytes = static_cast<size_t>(smem);
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n < 1) return cudaErrorInvalidConfiguration;
      max_pairs[dev] = n;
    }
    if (q.sched.grid > max_pairs[dev]) q.sched.grid = max_pairs[dev];
    static const bool pdl = [] {
      const char* v = std::getenv("HM_PDL");
      return !(v && v[0] == '0');
    }();
    cfg.gridDim = dim3(2u * static_cast<unsigned>(q.sched.grid));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, q);
  }
}

template <int WK, bool MOE>
cudaError_t launch_bt(const F16Params& p, int tile_m, cudaStream_t st) {
  switch (tile_m) {
    case 16: return launch_one<16, WK, MOE>(p, st);
    case 32: return launch_one<32, WK, MOE>(p, st);
    case 64: return launch_one<64, WK, MOE>(p, st);
    case 128:
      if constexpr (!MOE)
        if (p.pair) return launch_one<128, WK, MOE, false, true>(p, st);
      return launch_one<128, WK, MOE>(p, st);
    case 192:
      if constexpr (!MOE) return launch_one<192, WK, MOE>(p, st);
      return cudaErrorInvalidValue;
    case 256:
      if constexpr (WK != 8) {   // INT8 stops at 192
        if constexpr (!MOE)
          if (p.pair) return launch_one<256, WK, MOE, false, true>(p, st);
        return p.a_tmem1 ? launch_one<256, WK, MOE, true>(p, st) : launch_one<256, WK, MOE, false>(p, st);
      }
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Per-format entry points, each defined in its own translation unit so that the three sets of
// kernel instantiations compile in parallel.
cudaError_t launch_f16_mxfp4(const F16Params& p, int tile_m, bool moe, cudaStream_t st);
cudaError_t launch_f16_mxint4(const F16Params& p, int tile_m, bool moe, cudaStream_t st);
cudaError_t launch_f16_int4g(const F16Params& p, int tile_m, bool moe, cudaStream_t st);
cudaError_t launch_f16_int8(const F16Params& p, int tile_m, bool moe, cudaStream_t st);

}  // namespace hm
