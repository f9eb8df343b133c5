// W4A16 GEMM for decode-sized M (up to 16 tokens) on the tcgen05 tensor cores:
// Y[M,N] = X[M,K] * dequant(W)^T, dense or grouped MoE, INT4 weights (groups of 128, optional u4
// zero-points).
//
// The product and restore rule are those of the explainer page "vLLM Humming은 4비트를 어떻게
// 계산하나" (section "4비트 값에는 스케일이라는 해석 규칙이 붙는다": the restored weight is
// bf16((u - z) * s); section "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다": with few
// tokens every weight byte feeds only a few multiply-adds, so the kernel must stream and restore
// the weights as fast as HBM delivers them). The restored weights are exactly the oracle's, and
// every 128-K block of them goes through the tensor core into one fp32 accumulator per output
// tile and issuing thread.
//
// Why tcgen05 here: restoring a 128x128 unit costs every kernel the same CUDA-core work (one shift,
// one lop3, one bf16x2 subtract and one multiply per pair of weights); the warp-level MMA adds
// 64 m16n8k16 instructions per unit per SM on top, and on this GPU they are the bound (measured:
// ~3.8 TB/s with the restore removed). A tcgen05 MMA takes the whole 128-row unit for 16 tokens in
// 8 instructions issued by one thread, off the warps' issue slots.
//
//  * Work: the packed 128x128 units are cut into one contiguous range per CTA (the stream-K split of
//    the decode planner); the units of one output tile in a range form a segment.
//  * Roles (persistent CTA per SM, 20 warps): warp 0 loads one unit per stage (its weights by one
//    bulk copy, its 16 activation rows by one 3-D TMA box, 128-byte swizzled as the MMA's B
//    operand); three dequant groups of 4 warps take units i % 3, each thread restoring its own
//    weight row (one TMEM lane) into a ring of 6 TMEM slots of 64 columns (the MMA's A operand);
//    three issuing threads take units i % 3 (an issuing thread waits for its MMAs to drain at its
//    next shared-memory access, so several of them keep the tensor core fed), each accumulating
//    its units of a segment into its own TMEM accumulator (double-buffered); 4 epilogue warps add
//    the accumulators of a segment in issuer order (deterministic), then store Y or hand the tile
//    off.
//  * Shared tiles: fixed owner (the CTA holding the tile's first k-block); contributors store fp32
//    partials [CTA][16 tokens][128 rows] and add to the owner's counter; the owner waits (bounded),
//    adds them in CTA order and writes Y.
//  * Every mbarrier wait is bounded; the producer drains its copies and each issuer its MMAs before
//    the CTA frees TMEM and exits; PDL as in the other kernels.
#include <cuda_bf16.h>

#include "hm_dequant.cuh"
#include "hm_device.cuh"
#include "hm_f16_common.cuh"
#include "hm_kernels.h"
#include "hm_layout.h"
#include "hm_sched.cuh"

namespace hm {
namespace {

constexpr int kTcIss = 3;                   // issuing threads (one per warp): unit i goes to i % 3
constexpr int kTcGroups = 3;                // dequant groups of 4 warps: unit i goes to i % 3
constexpr int kTcSlots = 6;                 // TMEM slots of restored weights (64 columns each): i % 6
constexpr int kTcIss0 = 1;                  // warps: 0 producer, 1-3 issuers, 4-15 dequant, 16-19 epilogue
constexpr int kTcDq0 = kTcIss0 + kTcIss;
constexpr int kTcEpi0 = kTcDq0 + 4 * kTcGroups;
constexpr int kTcThreads = 32 * (kTcEpi0 + 4);
constexpr uint32_t kTcAccCol0 = kTcSlots * 64;   // accumulators [issuer][buffer], 16 columns each
constexpr uint32_t kTcCols = 512;
static_assert(kTcAccCol0 + 2 * kTcIss * kGemvMoeTokens <= kTcCols, "TMEM budget");
// Every barrier has one waiting role instance per use, which waits for its uses in order (an
// mbarrier parity wait cannot tell a phase two uses back from the one it waits for): a TMEM slot and
// a load stage always serve the same dequant group and the same issuer.
static_assert(kTcSlots % kTcGroups == 0 && kTcSlots % kTcIss == 0, "slot -> one group, one issuer");

template <int WB, bool MOE>
struct TcShape {
  static constexpr int kMT = kGemvMoeTokens;        // token rows of a tile (MMA N)
  static constexpr int kXUnit = 2 * kMT * 128;      // one unit's activations: [2 x 64 K][16 rows][128 B]
  static constexpr int kWArea = (WB + 1023) / 1024 * 1024;
  static constexpr int kStage = kWArea + kXUnit;    // one unit per stage
  static constexpr int kMoeBytes = MOE ? 2 * (kGemvMoeMaxExperts + 1) * 4 : 0;
  static constexpr int kFixedNoBars = 64 + kMoeBytes + 1024;   // misc, MoE arrays, alignment slack
  static constexpr int kSFit = (232448 - kFixedNoBars - 512) / kStage;
  static constexpr int kS = (kSFit > 16 ? 16 : kSFit) / 3 * 3;   // a multiple of the groups and issuers (3)
  static constexpr int kBarOff = kS * kStage;
  static constexpr int kNumBars = 2 * kS + 2 * kTcSlots + 4 * kTcIss + kTcIss;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kMoeOff = kMiscOff + 64;
  static constexpr int kSmem = kMoeOff + kMoeBytes + 1024;
  static_assert(kS >= 3 && kS % kTcGroups == 0 && kS % kTcIss == 0, "load stages: depth; stage -> one group, one issuer");
  static_assert(kWArea % 1024 == 0 && kStage % 1024 == 0, "activation boxes 1024-byte aligned (128-byte swizzle)");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

template <int WK, bool MOE>
__global__ void __launch_bounds__(kTcThreads, 1) tcdec_kernel(const __grid_constant__ F16Params p) {
  static_assert(WK == 0, "INT4 groups of 128");
  using S = TcShape<8704, MOE>;
  constexpr int SL = S::kS;
  constexpr int MT = S::kMT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);   // [stage] unit + activations landed
  uint64_t* empty = full + SL;                                        // [stage] its 4 dequant warps + issuer done
  uint64_t* a_full = empty + SL;                                      // [slot] restored weights in TMEM (4 warps)
  uint64_t* a_empty = a_full + kTcSlots;                              // [slot] MMAs reading it done (commit)
  uint64_t* acc_full = a_empty + kTcSlots;                            // [issuer][buffer] segment's MMAs done
  uint64_t* acc_empty = acc_full + 2 * kTcIss;                        // [issuer][buffer] epilogue read it (4 warps)
  uint64_t* drain = acc_empty + 2 * kTcIss;                           // [issuer] all of its MMAs done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + S::kMiscOff + 4);
  volatile uint32_t* hz_sh = abort_flag + 1;
  int32_t* mtpre = reinterpret_cast<int32_t*>(smem + S::kMoeOff);      // MoE: tile prefix [E+1]
  int32_t* moffs = mtpre + kGemvMoeMaxExperts + 1;                      // MoE: expert offsets [E+1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int32_t kb_total = p.sched.kb_total;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int s = 0; s < SL; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4 + 1);
    }
    for (int s = 0; s < kTcSlots; ++s) {
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < 2 * kTcIss; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    for (int q = 0; q < kTcIss; ++q) mbar_init(&drain[q], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // The (first) weight's header decides whether the units carry zero-points; every weight used
    // must agree with it and with the call's (fmt, N, K). (MoE: the expert pointers may come from
    // the previous kernel.)
    if (MOE) pdl_wait();
    const uint8_t* first_w = (MOE && p.packed_list != nullptr) ? p.packed_list[0] : p.packed;
    const PackedHeader hdr = *reinterpret_cast<const PackedHeader*>(first_w);
    *hz_sh = hdr.has_zero == 1u ? 1u : 0u;
    if (!(hdr.magic == kMagic && static_cast<int32_t>(hdr.fmt) == p.fmt && hdr.n == p.n && hdr.k == p.k)) {
      atomicOr(p.err, kErrHeader);
      *abort_flag = 1u;
    }
  }
  if (warp == kTcIss0) tmem_alloc(tmem_slot, kTcCols);
  if (MOE && warp == kTcEpi0) {
    // Every expert's header, then the offsets -> token tiles of 16 rows per expert x weight tiles,
    // exclusive prefix; a mismatch or malformed offsets abort every CTA before any weight is read.
    const bool list = p.packed_list != nullptr;
    if (list) pdl_wait();
    const uint32_t hz0 = reinterpret_cast<const PackedHeader*>(list ? p.packed_list[0] : p.packed)->has_zero;
    bool bad_hdr = false;
    for (int e = lane; e < p.num_experts; e += 32) {
      const uint8_t* w = list ? p.packed_list[e] : p.packed + static_cast<size_t>(e) * p.expert_stride;
      bad_hdr |= !header_ok(w, p, hz0 == 1u ? 1u : 0u);
    }
    pdl_wait();
    moe_tile_prefix<MT>(p, moffs, mtpre, abort_flag, lane);
    if (__any_sync(0xffffffffu, bad_hdr) && lane == 0) {
      atomicOr(p.err, kErrHeader);
      *abort_flag = 1u;
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // This CTA's range of the (tile, k-block) space (MoE: only the first `total` CTAs take units when
  // there are fewer units than CTAs, so that every CTA between a shared tile's owner and its last
  // contributor holds a part of it).
  const int64_t total = static_cast<int64_t>(MOE ? mtpre[p.num_experts] : p.sched.num_tiles) * kb_total;
  const int32_t grid = MOE ? static_cast<int32_t>(total < p.sched.grid ? total : p.sched.grid) : p.sched.grid;
  const bool idle = static_cast<int32_t>(blockIdx.x) >= grid;
  const int32_t u0 = idle ? 0 : static_cast<int32_t>(sk_start(blockIdx.x, total, grid));
  const int32_t u1 = idle ? 0 : static_cast<int32_t>(sk_start(blockIdx.x + 1, total, grid));
  const int32_t n_units = u1 - u0;
  const int32_t tile0 = u0 / kb_total, kb0 = u0 - tile0 * kb_total;
  if (threadIdx.x == 0) pdl_launch_dependents();
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  const bool aborted_early = *abort_flag != 0u;
  const uint32_t has_zero = *hz_sh;
  const uint32_t kUnit = has_zero ? kUnitInt4Zp : kUnitInt4;
  auto tile_info = [&](int32_t tile) -> TileInfo { return decode_tile<MT, MOE>(p, tile, mtpre, moffs, kUnit); };

  if (aborted_early) {
    // header or offsets rejected: nothing was issued
  } else if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // Stage i % SL holds unit i of the range: its weights (one bulk copy) and its activation block
    // (one 3-D box of 2 x 64 K, 16 token rows).
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    // (MoE: the unit's tile is decoded once per tile: `cur` caches it for the running unit)
    int32_t cur_tile = -1;
    TileInfo cur{};
    auto issue = [&](int i, bool weights, bool acts) {
      const int st = i % SL;
      uint8_t* sw = smem + st * S::kStage;
      const int32_t t = tile0 + (kb0 + i) / kb_total, kb = (kb0 + i) % kb_total;
      if (MOE && t != cur_tile) {
        cur = tile_info(t);
        cur_tile = t;
      }
      if (weights) {
        mbar_arrive_expect_tx(&full[st], kUnit + S::kXUnit);
        const uint8_t* src = MOE ? cur.wbase + static_cast<size_t>(kb) * kUnit
                                 : p.packed + kHeaderBytes + static_cast<size_t>(u0 + i) * kUnit;
        bulk_g2s(sw, src, kUnit, &full[st], pol_w);
      }
      if (acts) tma_3d_g2s(sw + S::kWArea, &p.tmap_x, 0, MOE ? cur.m0 : 0, 2 * kb, &full[st], pol_x);
    };
    const int first = n_units < SL ? n_units : SL;
    // Start-up, one stage per lane: the weights before waiting for the previous kernel (weights are
    // never written by another kernel; MoE tile decoding waited already), then the activations.
    if (lane < first) issue(lane, true, false);
    if (lane == 0) prefetch_tmap(&p.tmap_x);
    pdl_wait();
    if (lane < first) issue(lane, false, true);
    __syncwarp();
    if (lane == 0) {
      int issued = first;
      for (int i = first; i < n_units; ++i) {
        if (!mbar_wait(&empty[i % SL], static_cast<uint32_t>(i / SL - 1) & 1u, wc)) break;
        issue(i, true, true);
        issued = i + 1;
      }
      // nothing may still be landing in shared memory when the CTA exits
      for (int i = issued - SL < 0 ? 0 : issued - SL; i < issued; ++i)
        drain_wait(&full[i % SL], static_cast<uint32_t>(i / SL) & 1u, p.timeout_ns);
    }
  } else if (warp < kTcDq0) {
    // ---------------------------------------------------------------- MMA issuers
    // Issuer q takes units i = q, q + 3, ... Its units of a segment accumulate into its buffer
    // acc[q][c & 1] (c = its segments so far): the first MMA of its first unit in the segment
    // starts from zero; the commit after its last unit tells the epilogue. Each unit's commits
    // free its TMEM slot and (with its dequant group's arrivals) its load stage.
    const int q = warp - kTcIss0;
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, MT);
      uint32_t c = 0;   // this issuer's segments so far
      for (int i = q; i < n_units; i += kTcIss) {
        const int st = i % SL;
        if (!mbar_wait(&full[st], static_cast<uint32_t>(i / SL) & 1u, wc)) break;
        const int kbi = (kb0 + i) % kb_total;
        // this issuer's previous / next unit lies outside the unit's segment
        const bool seg_first = i < kTcIss || kbi < kTcIss;
        const bool seg_last = i + kTcIss > n_units - 1 || kbi + kTcIss > kb_total - 1;
        const uint32_t buf = 2 * q + (c & 1u);
        if (seg_first && !mbar_wait(&acc_empty[buf], ((c >> 1) & 1u) ^ 1u, wc)) break;
        const int s = i % kTcSlots;
        if (!mbar_wait(&a_full[s], static_cast<uint32_t>(i / kTcSlots) & 1u, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem + kTcAccCol0 + buf * MT;
        const uint32_t a = tmem + s * 64;
        const uint32_t xb = smem_u32(smem + st * S::kStage + S::kWArea);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bd = sdesc_sw128(xb + (k >> 2) * (MT * 128) + (k & 3) * 32);
          mma_bf16_ta(d, a + 8 * k, bd, idesc, (seg_first && k == 0) ? 0u : 1u);
        }
        tc_commit(&a_empty[s]);
        tc_commit(&empty[st]);
        if (seg_last) {
          tc_commit(&acc_full[buf]);
          ++c;
        }
      }
      // all tcgen05 work of this thread has completed once `drain` flips
      tc_commit(&drain[q]);
      drain_wait(&drain[q], 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < kTcEpi0) {
    // ---------------------------------------------------------------- dequant warps
    // Group g restores units i = g, g + 3, ...; thread `lane` of warp w owns weight row r = 32 (w % 4) +
    // lane, which is its TMEM lane: it reads the row's 64 code bytes, scale and zero-point, forms
    // the 128 restored weights bf16((u - z) s) as 64 bf16x2 columns (k, k + 1) and stores them in
    // the unit's slot.
    const int g = (warp - kTcDq0) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    for (int i = g; i < n_units; i += kTcGroups) {
      const int st = i % SL;
      if (!mbar_wait(&full[st], static_cast<uint32_t>(i / SL) & 1u, wc)) break;
      const int s = i % kTcSlots;
      if (!mbar_wait(&a_empty[s], (static_cast<uint32_t>(i / kTcSlots) & 1u) ^ 1u, wc)) break;
      const uint32_t wsa = smem_u32(smem + st * S::kStage);
      uint4 cw[4];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) cw[cc] = ld_shared_v4(wsa + cc * 2048 + r * 16);
      uint16_t sb;
      asm volatile("ld.shared.b16 %0, [%1];" : "=h"(sb) : "r"(wsa + kUnitCodes + 2 * r));
      uint32_t z = 8u;
      if (has_zero) {
        uint16_t zb;
        asm volatile("ld.shared.u8 %0, [%1];" : "=h"(zb) : "r"(wsa + kUnitInt4 + (r >> 1)));
        z = (static_cast<uint32_t>(zb) >> (4 * (r & 1))) & 0xFu;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);   // this unit's bytes are in registers
      const __nv_bfloat162 zz = int4_zero_pair(z), ss = bf16_pair(sb);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t a_regs[32];   // 64 restored K of this row as bf16x2, in K order
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
          const uint4 v = cw[2 * half + ci];
          const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint32_t o[4];
            dq_int4_word(words[t], zz, ss, o);
#pragma unroll
            for (int e = 0; e < 4; ++e) a_regs[16 * ci + 4 * t + e] = o[e];
          }
        }
        tmem_st32(tmem + lane_base + s * 64 + half * 32, a_regs);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[s]);
    }
  } else {
    // ---------------------------------------------------------------- epilogue warps
    // Per segment: the accumulators of the issuers that had units in it, issuer 0 first; then Y,
    // or the fixed-owner hand-off of a tile shared with other CTAs.
    pdl_wait();   // Y, partials and counters may be in use by the previous kernel
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    uint32_t cnt[kTcIss] = {};
    int32_t a = 0;
    int32_t kb = kb0;
    int32_t tile = tile0;
    bool ok = true;
    while (ok && a < n_units) {
      const int32_t len = kb_total - kb < n_units - a ? kb_total - kb : n_units - a;
      float acc[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) acc[t] = 0.f;
#pragma unroll
      for (int q = 0; q < kTcIss; ++q) {
        if (len < kTcIss && (q - a % kTcIss + kTcIss) % kTcIss >= len) continue;   // issuer q had no unit here
        const uint32_t buf = 2 * q + (cnt[q] & 1u);
        if (!mbar_wait(&acc_full[buf], (cnt[q] >> 1) & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + kTcAccCol0 + buf * MT, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        ++cnt[q];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] += __uint_as_float(v[t]);
      }
      if (!ok) break;
      const TileInfo ti = tile_info(tile);
      const int64_t n = static_cast<int64_t>(ti.n0) + row;
      const int tok_end = MOE ? ti.m_end - ti.m0 : static_cast<int>(p.m);
      auto store_y = [&]() {
        if (n < p.n) {
#pragma unroll
          for (int t = 0; t < MT; ++t)
            if (t < tok_end) p.y[static_cast<size_t>(ti.m0 + t) * p.n + n] = __float2bfloat16_rn(acc[t]);
        }
      };
      if (kb == 0 && len == kb_total) {
        store_y();
      } else {
        const int64_t it0 = static_cast<int64_t>(tile) * kb_total;
        if (kb != 0) {
          // contributor: the tile's first k-block belongs to an earlier CTA
          const int64_t c_lo = sk_owner(it0, total, grid);
#pragma unroll
          for (int t = 0; t < MT; ++t)
            __stcg(p.partial + (static_cast<size_t>(blockIdx.x) * MT + t) * 128 + row, acc[t]);
          __syncwarp();
          if (lane == 0)
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(sk_flag(p.counters, c_lo, q4)) : "memory");
        } else {
          // owner: wait for the contributors, add their partials in CTA order, write Y
          const int64_t c_hi = sk_owner(it0 + kb_total - 1, total, grid);
          uint32_t* ctr = sk_flag(p.counters, blockIdx.x, q4);
          if (!sk_wait(ctr, static_cast<uint32_t>(c_hi - blockIdx.x), wc)) break;
          for (int64_t c = blockIdx.x + 1; c <= c_hi; ++c) {
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[t] += __ldcg(p.partial + (static_cast<size_t>(c) * MT + t) * 128 + row);
          }
          store_y();
          __syncwarp();
          if (lane == 0) *ctr = 0u;   // for the next call
        }
      }
      a += len;
      kb += len;
      if (kb == kb_total) {
        kb = 0;
        ++tile;
      }
    }
  }
  __syncwarp();
  __syncthreads();
  if (warp == kTcIss0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcCols);
  }
}

template <int WK, bool MOE>
cudaError_t launch_tc(const F16Params& p, cudaStream_t st) {
  using S = TcShape<8704, MOE>;
  auto kern = tcdec_kernel<WK, MOE>;
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return launch_pdl(kern, p.sched.grid, kTcThreads, S::kSmem, st, p);
}

}  // namespace

bool tcdec_serves(int32_t fmt) { return fmt == kW4A16Int4; }

int tcdec_stages() { return TcShape<8704, false>::kS; }

cudaError_t launch_tcdec(const F16Params& p, bool moe, cudaStream_t st) {
  if (!tcdec_serves(p.fmt) || p.k % 128 != 0 || (!moe && (p.m < 1 || p.m > kGemvMoeTokens)) ||
      (moe && (p.num_experts < 1 || p.num_experts > kGemvMoeMaxExperts)))
    return cudaErrorInvalidValue;
  return moe ? launch_tc<0, true>(p, st) : launch_tc<0, false>(p, st);
}

}  // namespace hm
