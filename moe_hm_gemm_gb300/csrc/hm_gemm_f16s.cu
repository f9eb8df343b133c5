// W4A16 GEMM for small token tiles (tile_m 16 or 32) with INT4 weights, on tcgen05:
// Y[M,N] = X[M,K] * dequant(W)^T, dense or grouped MoE.
//
// Same product as the general W4A16 kernel (the explainer page's linear layer, "vLLM Humming은
// 4비트를 어떻게 계산하나", section "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다",
// with W restored by the rule of section "4비트 값에는 스케일이라는 해석 규칙이 붙는다"), arranged
// for decode-sized M, where every weight byte is used by at most 32 tokens and the kernel must
// keep pace with HBM:
//  * the group scale is applied once per 128-K block to the fp32 partial sum of that block
//    rather than to each weight: sum_k x*(u-z)*s = s * sum_k x*(u-z) within a group. The
//    dequant warps therefore only form the exact integers u - z in bf16 (one shift, one lop3 and
//    one bf16x2 subtract per pair of weights), and each block accumulates into its own TMEM
//    accumulator taken from a ring; the epilogue warps add s * P_block in fp32, block by block,
//    in k order (deterministic);
//  * a thread that issues tcgen05.mma waits ~50 cycles per instruction and then stalls at its next
//    shared-memory access until its MMAs drain, while the tensor core takes small-N MMAs from
//    several threads far faster. So the two 128-K blocks of each half load stage form a pair,
//    pairs go round-robin to NI issuing warps (3 for tile_m 16, 2 for 32, as TMEM allows), and an
//    issuer waits once per pair and then issues its 16 MMAs back to back;
//  * every TMEM slot (restored weights, block accumulator) and its barriers belong to one
//    (issuer, dequant group) pair, so each barrier has one producer and one consumer that use it
//    strictly in turn: every wait is for the next phase of that slot, never one further ahead;
//  * everything else (persistent CTA per SM, TMA bulk loads of packed 128x128 units, weights
//    restored into TMEM as the MMA's A operand, stream-K for tiles fewer than SMs, PDL, bounded
//    waits) follows the general kernel.
#include <cuda_bf16.h>

#include "hm_dequant.cuh"
#include "hm_device.cuh"
#include "hm_f16_common.cuh"
#include "hm_kernels.h"
#include "hm_layout.h"
#include "hm_sched.cuh"

namespace hm {
namespace {

constexpr int kSIssMax = 3;                  // MMA issuing warps (tile_m 32 uses two of them)
constexpr int kSDqGroup = 4;                 // warps per dequant group (one per TMEM lane quarter)
constexpr int kSDqWarps = 2 * kSDqGroup;     // two groups take alternate 128-K blocks
constexpr int kSMma0 = 1;                    // warps: 0 producer, 1-3 MMA, 4-11 dequant, 12-15 epilogue
constexpr int kSDq0 = kSMma0 + kSIssMax;
constexpr int kSEpi0 = kSDq0 + kSDqWarps;
constexpr int kSThreads = 32 * (kSEpi0 + 4);   // 16 warps: 4 per SM sub-partition, 128 registers each

template <int BT>
struct SShape {
  static constexpr int kG = f16_group_of(BT);       // 128-K blocks per load stage (4)
  static constexpr int kNI = BT == 16 ? 3 : 2;      // issuing warps
  static constexpr int kNS = 2 * kNI;               // slots: (issuer, dequant group)
  static constexpr uint32_t kACol0 = kNS * BT;      // block accumulators at [0, kNS*BT), then A slots
  static constexpr int kXStage = kG * BT * 128 * 2;
  static constexpr int kWStage = kG * kUnitInt4Zp;
  static constexpr int kMetaBytes = kNS * 2 * 128 * 4;   // group scales: [slot][use parity][row]
  static constexpr int kSLFit = (212 * 1024 - kMetaBytes) / (kXStage + kWStage);
  static constexpr int kSL = kSLFit > 16 ? 16 : kSLFit;
  static constexpr int kXOff = 0;
  static constexpr int kWOff = kXOff + kSL * kXStage;
  static constexpr int kMetaOff = kWOff + kSL * kWStage;
  static constexpr int kBarOff = kMetaOff + kMetaBytes;
  static constexpr int kNumBars = 3 * kSL + 6 * kNS + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kMoeOff = kMiscOff + 32;
  static constexpr int smem_bytes(int experts) { return 1024 + kMoeOff + 8 * (experts + 1); }
  static_assert(BT == 16 || BT == 32, "small token tiles only");
  static_assert(kSL >= 3, "load pipeline depth (the issuers' skipped stages rely on it)");
  static_assert(kACol0 + kNS * 64 <= 512, "TMEM budget");
  static_assert(kNI <= kSIssMax, "issuing warps");
};

// Walks the block sequence of a CTA's schedule the way every role does: segments, load stages of
// up to kG blocks, and pairs of blocks (j, j + 1) within a stage; pair index `pair` runs over the
// whole range. Block j of the current stage belongs to dequant group (seq + j) & 1 and to issuer
// pair % NI.
struct PairWalk {
  int seq = 0;       // running block index at the current stage's start
  int pair0 = 0;     // pair index of the current stage's first pair
  __device__ __forceinline__ int pair_of(int j) const { return pair0 + (j >> 1); }
  __device__ __forceinline__ void next_stage(int g) {
    seq += g;
    pair0 += (g + 1) >> 1;
  }
};

template <int BT, bool MOE>
__global__ void __launch_bounds__(kSThreads, 1) f16s_gemm_kernel(const __grid_constant__ F16Params p) {
  using S = SShape<BT>;
  constexpr int SL = S::kSL;
  constexpr int NI = S::kNI;
  constexpr int NS = S::kNS;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* full_w = bars;
  uint64_t* full_x = full_w + SL;
  uint64_t* empty_l = full_x + SL;
  uint64_t* full_a = empty_l + SL;       // [slot] restored weights in TMEM (4 dequant warps)
  uint64_t* empty_a = full_a + NS;       // [slot] their MMAs done (commit)
  uint64_t* acc_full = empty_a + NS;     // [slot] block accumulator ready (commit)
  uint64_t* acc_empty = acc_full + NS;   // [slot] drained by the epilogue (4 warps)
  uint64_t* meta_full = acc_empty + NS;  // [slot][use parity] group scale written (4 dequant warps)
  uint64_t* drain = meta_full + 2 * NS;
  float* meta = reinterpret_cast<float*>(smem + S::kMetaOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + S::kMiscOff + 4);
  volatile uint32_t* hz_sh = reinterpret_cast<volatile uint32_t*>(smem + S::kMiscOff + 8);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + S::kMoeOff);
  int32_t* offs = prefix + (MOE ? p.num_experts + 1 : 0);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (MOE) {
    // The MoE prefix warp may raise the abort flag while thread 0 is still setting up: clear the
    // flag before any role runs, so that a raised flag is never overwritten.
    if (threadIdx.x == 0) *abort_flag = 0u;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    trace_mark(p.trace, 0);
    if (MOE) pdl_wait();   // expert pointers may come from the previous kernel
    const uint8_t* first = (MOE && p.packed_list != nullptr) ? p.packed_list[0] : p.packed;
    const PackedHeader hdr = *reinterpret_cast<const PackedHeader*>(first);
    for (int s = 0; s < SL; ++s) {
      mbar_init(&full_w[s], 1);
      mbar_init(&full_x[s], 1);
      mbar_init(&empty_l[s], 4 + kSDqWarps);   // epilogue warps (X read by the MMAs) + dequant warps (W)
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_a[s], kSDqGroup);
      mbar_init(&empty_a[s], 1);
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
      mbar_init(&meta_full[2 * s], kSDqGroup);
      mbar_init(&meta_full[2 * s + 1], kSDqGroup);
    }
    mbar_init(drain, NI);
    fence_barrier_init();
    if (!MOE) *abort_flag = 0u;
    *hz_sh = hdr.has_zero == 1u ? 1u : 0u;
    if (!(hdr.magic == kMagic && static_cast<int32_t>(hdr.fmt) == p.fmt && hdr.n == p.n && hdr.k == p.k)) {
      atomicOr(p.err, kErrHeader);
      *abort_flag = 1u;
    }
  }
  if (warp == kSMma0) tmem_alloc(tmem_slot, 512);
  if (MOE && warp == kSDq0) {
    pdl_wait();   // the offsets may be written by the previous kernel
    moe_tile_prefix<BT>(p, offs, prefix, abort_flag, lane);
  }
  __syncthreads();
  tc_fence_after();
  const int32_t num_tiles = MOE ? prefix[p.num_experts] : p.sched.num_tiles;
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  SchedIter sched;
  sched.init(p.sched, num_tiles, blockIdx.x);
  const int kb_total = p.sched.kb_total;
  const bool aborted_early = *abort_flag != 0u;
  const uint32_t has_zero = *hz_sh;
  if (threadIdx.x == 0) {
    trace_mark(p.trace, 1);
    pdl_launch_dependents();
  }
  const uint32_t kUnit = has_zero ? kUnitInt4Zp : kUnitInt4;
  const bool reuse_w = MOE || p.num_m_tiles > 1;

  if (aborted_early) {
    // nothing to do: fall through to teardown
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tmap_x);
      const uint64_t pol_w = reuse_w ? policy_evict_last() : policy_evict_first();
      const uint64_t pol_x = reuse_w ? policy_evict_normal() : policy_evict_last();
      const uint8_t* last_checked = nullptr;
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
      auto issue_w = [&](int idx, const TileInfo& t, int kb, int g) {
        const int slot = idx % SL;
        const uint32_t bytes = static_cast<uint32_t>(g) * kUnit;
        mbar_arrive_expect_tx(&full_w[slot], bytes);
        bulk_g2s(smem + S::kWOff + slot * S::kWStage, t.wbase + static_cast<size_t>(kb) * kUnit, bytes,
                 &full_w[slot], pol_w);
      };
      auto issue_x = [&](int idx, const TileInfo& t, int kb) {
        const int slot = idx % SL;
        mbar_arrive_expect_tx(&full_x[slot], S::kXStage);   // the whole box lands (zero-filled past M, K)
        tma_3d_g2s(smem + S::kXOff + slot * S::kXStage, &p.tmap_x, 0, t.m0, 2 * kb, &full_x[slot], pol_x);
        if (idx == 0) trace_mark(p.trace, 2);
      };
      // Start-up: stage 0's weights before the wait for the previous kernel (they do not depend
      // on it), then the activation tiles of the first SL stages ahead of the remaining weights
      // (an SM's copies complete roughly in issue order).
      int issued_w = 0, issued_x = 0;
      bool ok = true;
      if (!MOE) {
        SchedIter pf = sched;
        Segment ps;
        if (pf.next(ps)) {
          issue_w(0, decode_tile<BT, MOE>(p, ps.tile, prefix, offs, kUnit), ps.kb0, min(S::kG, ps.kb1 - ps.kb0));
          issued_w = 1;
        }
      }
      pdl_wait();
      {
        SchedIter pf = sched;
        Segment ps;
        int idx = 0;
        while (idx < SL && pf.next(ps)) {
          const TileInfo t = decode_tile<BT, MOE>(p, ps.tile, prefix, offs, kUnit);
          for (int kb = ps.kb0; kb < ps.kb1 && idx < SL; kb += S::kG, ++idx) issue_x(idx, t, kb);
        }
        issued_x = idx;
        pf = sched;
        idx = 0;
        while (idx < issued_x && pf.next(ps)) {
          const TileInfo t = decode_tile<BT, MOE>(p, ps.tile, prefix, offs, kUnit);
          if (!checked(t)) { ok = false; break; }
          for (int kb = ps.kb0; kb < ps.kb1 && idx < issued_x; kb += S::kG, ++idx)
            if (idx >= issued_w) issue_w(idx, t, kb, min(S::kG, ps.kb1 - kb));
        }
        if (ok) issued_w = issued_x;
      }
      int idx = 0;
      int ls = 0;
      uint32_t lph = 0;
      Segment seg;
      while (ok && sched.next(seg)) {
        const TileInfo t = decode_tile<BT, MOE>(p, seg.tile, prefix, offs, kUnit);
        if (!checked(t)) break;
        for (int kb = seg.kb0; kb < seg.kb1; kb += S::kG, ++idx) {
          if (idx >= issued_x) {
            if (!mbar_wait(&empty_l[ls], lph ^ 1u, wc)) { ok = false; break; }
            issue_w(idx, t, kb, min(S::kG, seg.kb1 - kb));
            issue_x(idx, t, kb);
            issued_x = issued_w = idx + 1;
          }
          if (++ls == SL) { ls = 0; lph ^= 1u; }
        }
      }
      trace_mark(p.trace, 3);
      if (*abort_flag) {
        for (int i = issued_x > SL ? issued_x - SL : 0; i < issued_x; ++i)
          drain_wait(&full_x[i % SL], static_cast<uint32_t>(i / SL) & 1u, 100000000ull);
        for (int i = issued_w > SL ? issued_w - SL : 0; i < issued_w; ++i)
          drain_wait(&full_w[i % SL], static_cast<uint32_t>(i / SL) & 1u, 100000000ull);
      }
    }
  } else if (warp < kSDq0) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer `is` takes pairs pair % NI == is. For each block of the pair (dequant group g =
    // block & 1, slot is*2 + g): wait until the slot's accumulator was drained and its restored
    // weights are in TMEM; then one fence and all of the pair's MMAs (each block into its own
    // accumulator, from zero); then the commits. The issuers do not release load stages: the
    // epilogue does, once it has seen the MMAs of a stage's last block complete.
    if (lane == 0 && warp - kSMma0 < NI) {
      const int is = warp - kSMma0;
      constexpr uint32_t idesc = idesc_bf16(128, BT);
      uint32_t par = 0u;   // bit g: parity of the number of uses of slot (is, g) so far
      int ls = 0;
      uint32_t lph = 0;
      PairWalk pw;
      bool first = true;
      Segment seg;
      bool ok = true;
      while (ok && sched.next(seg)) {
        for (int kb0 = seg.kb0; kb0 < seg.kb1 && ok; kb0 += S::kG) {
          const int g = min(S::kG, seg.kb1 - kb0);
          bool have_x = false;
          for (int j0 = 0; j0 < g && ok; j0 += 2) {
            if (pw.pair_of(j0) % NI != is) continue;
            if (!have_x) {
              if (!mbar_wait(&full_x[ls], lph, wc)) { ok = false; break; }
              have_x = true;
            }
            const int nb = min(2, g - j0);
            for (int u = 0; u < nb && ok; ++u) {
              const int gr = (pw.seq + j0 + u) & 1;
              const int sl = 2 * is + gr;
              const uint32_t ph = (par >> gr) & 1u;
              ok = mbar_wait(&acc_empty[sl], ph ^ 1u, wc) && mbar_wait(&full_a[sl], ph, wc);
              if (ok) trace_stage(p.trace, 3, pw.seq + j0 + u);
            }
            if (!ok) break;
            tc_fence_after();
            if (first && is == 0) trace_mark(p.trace, 6);
            first = false;
            for (int u = 0; u < nb; ++u) {
              const int sl = 2 * is + ((pw.seq + j0 + u) & 1);
              const uint32_t d = tmem + sl * BT;
              const uint32_t a_t = tmem + S::kACol0 + sl * 64;
              const uint32_t x_base = smem_u32(smem + S::kXOff + ls * S::kXStage) + (j0 + u) * (2 * BT * 128);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint64_t bd = sdesc_sw128(x_base + (k >> 2) * (BT * 128) + (k & 3) * 32);
                mma_bf16_ta(d, a_t + 8 * k, bd, idesc, k > 0 ? 1u : 0u);
              }
              trace_stage(p.trace, 5, pw.seq + j0 + u);
            }
            for (int u = 0; u < nb; ++u) {
              const int gr = (pw.seq + j0 + u) & 1;
              tc_commit(&empty_a[2 * is + gr]);
              tc_commit(&acc_full[2 * is + gr]);
              par ^= 1u << gr;
            }
          }
          pw.next_stage(g);
          if (++ls == SL) { ls = 0; lph ^= 1u; }
        }
      }
      if (is == 0) trace_mark(p.trace, 7);
      // All tcgen05 work of this thread has completed once `drain` flips (one arrival per issuer).
      tc_commit(drain);
      drain_wait(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp < kSEpi0) {
    // ------------------------------------------------------------ dequant warps
    // Group grp restores the blocks with sequence index % 2 == grp; its warp for TMEM lane
    // quarter warp % 4 handles weight rows 32*(warp % 4) .. +31, one row per thread. A block goes
    // to the slot of its pair's issuer; the row's group scale goes to that slot's scale entry for
    // the use parity (published through meta_full) for the epilogue.
    const int dw = warp - kSDq0;
    const int grp = dw / kSDqGroup;
    const int r = 32 * (warp & 3) + lane;
    uint32_t par = 0u;   // bit i: parity of the number of uses of slot (issuer i, grp) so far
    int ls = 0;
    uint32_t lph = 0;
    PairWalk pw;
    bool first_dq = true;
    Segment seg;
    bool ok = true;
    while (ok && sched.next(seg)) {
      for (int kb0 = seg.kb0; kb0 < seg.kb1 && ok; kb0 += S::kG) {
        const int g = min(S::kG, seg.kb1 - kb0);
        const int j0 = ((pw.seq & 1) == grp) ? 0 : 1;
        // Every group waits for the stage to fill, even one with no block in it: its release must
        // not reach the slot's empty barrier before the slot's previous use is over.
        if (!mbar_wait(&full_w[ls], lph, wc)) { ok = false; break; }
        if (j0 >= g) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_l[ls]);
        }
        for (int jb = j0; jb < g; jb += 2) {
          const int bi = pw.seq + jb;
          const int iss = pw.pair_of(jb) % NI;
          const int sl = 2 * iss + grp;
          const uint32_t u = (par >> iss) & 1u;
          if (!mbar_wait(&empty_a[sl], u ^ 1u, wc)) { ok = false; break; }
          if (dw == 0 && first_dq) { trace_mark(p.trace, 4); first_dq = false; }
          if (dw % kSDqGroup == 0 && lane == 0) trace_stage(p.trace, 1, bi);
          const uint32_t wsa = smem_u32(smem + S::kWOff + ls * S::kWStage) + jb * kUnit;
          uint4 c[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) c[i] = ld_shared_v4(wsa + i * 2048 + r * 16);
          uint16_t sb;
          asm volatile("ld.shared.b16 %0, [%1];" : "=h"(sb) : "r"(wsa + kUnitCodes + 2 * r));
          uint32_t z = 8u;
          if (has_zero) {
            uint16_t zb;
            asm volatile("ld.shared.u8 %0, [%1];" : "=h"(zb) : "r"(wsa + kUnitInt4 + (r >> 1)));
            z = (static_cast<uint32_t>(zb) >> (4 * (r & 1))) & 0xFu;
          }
          const uint32_t z2 = bf16x2_bits(int4_zero_pair(z));
          meta[(sl * 2 + u) * 128 + r] = __uint_as_float(static_cast<uint32_t>(sb) << 16);
          __syncwarp();
          if (lane == 0) mbar_arrive(&meta_full[2 * sl + u]);
          if (jb + 2 >= g) {   // the stage's last block of this group is in registers: release it
            if (lane == 0) mbar_arrive(&empty_l[ls]);
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t a_regs[32];   // 64 restored K of this row as bf16x2, in K order
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const uint4 cc = c[2 * half + i];
              const uint32_t words[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t o[4];
                dq_int4_word_unscaled(words[j], z2, o);
#pragma unroll
                for (int t = 0; t < 4; ++t) a_regs[16 * i + 4 * j + t] = o[t];
              }
            }
            tmem_st32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + S::kACol0 + sl * 64 + half * 32,
                      a_regs);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (dw % kSDqGroup == 0 && lane == 0) trace_stage(p.trace, 2, bi);
          if (lane == 0) mbar_arrive(&full_a[sl]);
          par ^= 1u << iss;
        }
        pw.next_stage(g);
        if (++ls == SL) { ls = 0; lph ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    // Drain each block's accumulator as soon as its MMAs complete, scale it by the row's group
    // scale and add it to the segment's running fp32 sum (k order); store the segment at its end.
    // After a stage's last block, release the stage (its activation tile was read by the MMAs).
    pdl_wait();                          // Y, partials and counters may be in use by the previous kernel
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int row = 32 * q + lane;
    const int64_t total_it = static_cast<int64_t>(num_tiles) * kb_total;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    uint32_t par = 0u;        // bit sl: parity of the number of uses of slot sl so far
    uint32_t uses_meta = 0u;  // bit sl: parity of the number of uses of meta_full[sl][u] (every other use)
    int ls = 0;
    PairWalk pw;
    bool first_seg = true;
    bool ok = true;
    Segment seg;
    while (ok && sched.next(seg)) {
      float acc[BT];
#pragma unroll
      for (int j = 0; j < BT; ++j) acc[j] = 0.f;
      for (int kb0 = seg.kb0; kb0 < seg.kb1 && ok; kb0 += S::kG) {
        const int g = min(S::kG, seg.kb1 - kb0);
        for (int j = 0; j < g; ++j) {
          const int bi = pw.seq + j;
          const int sl = 2 * (pw.pair_of(j) % NI) + (bi & 1);
          const uint32_t u = (par >> sl) & 1u;
          if (!mbar_wait(&acc_full[sl], u, wc)) { ok = false; break; }
          tc_fence_after();
          if (row == 0 && first_seg && kb0 == seg.kb0 && j == 0) trace_mark(p.trace, 8);
          if (row == 0) trace_stage(p.trace, 0, bi);
          uint32_t v[BT];
#pragma unroll
          for (int j0 = 0; j0 < BT; j0 += 16)
            tmem_ld16(tmem + lane_base + sl * BT + j0, *reinterpret_cast<uint32_t(*)[16]>(v + j0));
          tmem_wait_ld();
          // Scale entries and their barriers are kept per use parity: the dequant warps may write
          // the slot's next scale before this one is read.
          if (!mbar_wait(&meta_full[2 * sl + u], (uses_meta >> sl) & 1u, wc)) { ok = false; break; }
          const float s = meta[(sl * 2 + u) * 128 + row];
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[sl]);
          par ^= 1u << sl;
          if (u) uses_meta ^= 1u << sl;   // both parity barriers of the slot have now been used once more
#pragma unroll
          for (int jj = 0; jj < BT; ++jj) acc[jj] = fmaf(s, __uint_as_float(v[jj]), acc[jj]);
        }
        if (!ok) break;
        if (lane == 0) mbar_arrive(&empty_l[ls]);
        if (++ls == SL) ls = 0;
        pw.next_stage(g);
      }
      if (!ok) break;
      const TileInfo t = decode_tile<BT, MOE>(p, seg.tile, prefix, offs, kUnit);
      store_segment<BT>(p, t, seg, kb_total, total_it, first_seg, q, lane, wc, acc);
      if (row == 0) trace_mark(p.trace, 9);
      first_seg = false;
    }
  }

  __syncwarp();  // reconverge lanes that skipped a single-thread role before the CTA barrier
  __syncthreads();
  if (warp == kSMma0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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

template <int BT, bool MOE>
cudaError_t launch_s(const F16Params& p, cudaStream_t st) {
  using S = SShape<BT>;
  auto kern = f16s_gemm_kernel<BT, MOE>;
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::smem_bytes(1024));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return launch_pdl(kern, p.sched.grid, kSThreads, S::smem_bytes(MOE ? p.num_experts : 0), st, p);
}

}  // namespace

int f16s_stages(int tile_m) { return tile_m <= 16 ? SShape<16>::kSL : SShape<32>::kSL; }

cudaError_t launch_f16s_gemm(const F16Params& p, int tile_m, bool moe, cudaStream_t st) {
  if (tile_m == 16) return moe ? launch_s<16, true>(p, st) : launch_s<16, false>(p, st);
  if (tile_m == 32) return moe ? launch_s<32, true>(p, st) : launch_s<32, false>(p, st);
  return cudaErrorInvalidValue;
}

}  // namespace hm
