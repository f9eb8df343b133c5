// Block-scaled GEMMs on tcgen05: the W4A8 (MXFP4 weights x per-token FP8 activations) and
// W4A4 (NVFP4 x NVFP4) formats named on the news page's format list (news.cocoloop.cn,
// section "하나의 라이브러리로 긴 포맷 목록을 포괄"), computing the explainer page's linear layer
// Y = X * W^T ("vLLM Humming은 4비트를 어떻게 계산하나", section "같은 가중치도 한 토큰과 많은
// 토큰에서 비용이 다르다") with both operands in their quantized form.
//
//  * W4A8: kind::mxf8f6f4.block_scale.scale_vec::1X. A = weight codes (e2m1), expanded by
//    TMA (16 x 4-bit packed -> 16-byte aligned) into one byte per code in shared memory;
//    B = e4m3 activations; A scales = the weight's E8M0 per 32 along K; B scales = 1
//    (E8M0 127); the per-token fp32 scale multiplies each output column in the epilogue:
//    Y[m,n] = s_tok[m] * sum_k e4m3(x[m,k]) * e2m1(w[n,k]) * 2^(e[n,k/32]-127).
//  * W4A4: kind::mxf4nvf4.block_scale.scale_vec::4X. A and B = packed e2m1 codes, scales
//    = e4m3 per 16 along K for both; the two fp32 tensor scales multiply in the epilogue.
//
// Scale factors are staged by a bulk copy into shared memory in 512-byte atoms (128 rows x 4
// scales, row r at byte (r%32)*16 + (r/32)*4) and moved to TMEM with
// tcgen05.cp.32x128b.warpx4, which puts row r's four scales in lane r%32 (every 32-lane
// group) of column r/32 of a 4-column slot; the MMA picks the byte with the scale-factor id
// (1X) or uses all four (4X). Persistent, two CTAs per SM (see MxShape): warp 0 loads, warp 1
// issues MMAs (and the scale copies), warps 2-5 drain TMEM.
//
// Grouped (MoE) variant: the rows arrive sorted by expert with device offsets [E+1] (the MoE
// paragraph of the explainer page's section "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다");
// the experts' packed weights lie back to back at a fixed stride, so one 3-D tensor map (K, N,
// expert) reaches every expert's codes and its scale atoms are found by address. One warp turns
// the offsets into a per-expert tile prefix in shared memory (tiles m-major within an expert, as
// in the W4A16 grouped kernel), checks every expert's header and keeps each expert's NVFP4 tensor
// scale. NVFP4 activation scale atoms are laid out per expert token tile (block = the tile's
// ordinal among all experts' token tiles), since an expert's rows need not start on a 128-row
// boundary.
#pragma once
#include <cuda_bf16.h>

#include "hm_device.cuh"
#include "hm_kernels.h"
#include "hm_layout.h"
#include "hm_sched.cuh"

namespace hm {
namespace {

// Warps: 0 loads, 1 issues MMAs, 2-5 drain TMEM; W4A4 adds warps 6 and 7, which copy the four
// weight and the four activation scale atoms of each 256-K block to TMEM (W4A8 has one copy per
// block, kept on the MMA thread).
template <bool NV>
constexpr int threads_of() { return NV ? 256 : 192; }
constexpr int kSfWarp = 6;
constexpr int kWTile = 128 * 128;  // weight stage: 128 rows x 128 bytes (swizzled)

// Two CTAs share each SM (kMxCtasPerSm): each has its own MMA-issuing thread, which a single
// thread per SM cannot keep up with at FP8/FP4 rates (it issues every scale copy and MMA and
// stalls at its next shared-memory access until its MMAs are under way), and while one CTA
// drains its accumulator the other keeps the tensor pipe busy. So each CTA takes half of the
// shared memory and at most 256 TMEM columns with a single accumulator.
template <int BT, bool NV, bool MOE = false>
struct MxShape {
  static constexpr int kXStage = BT * 128;                          // 128 bytes of K per row
  static constexpr int kSfaBytes = NV ? 4 * kAtomBytes : kAtomBytes;  // per stage
  static constexpr int kSfbBytes = NV ? 4 * kAtomBytes : 0;
  static constexpr int kStageBytes = kWTile + kXStage + kSfaBytes + kSfbBytes;
  static constexpr int kBudget = 108 * 1024;
  static constexpr int kSL = kBudget / kStageBytes > 8 ? 8 : kBudget / kStageBytes;
  static constexpr int kWOff = 0;
  static constexpr int kXOff = kWOff + kSL * kWTile;
  static constexpr int kSfaOff = kXOff + kSL * kXStage;
  static constexpr int kSfbOff = kSfaOff + kSL * kSfaBytes;
  static constexpr int kUnitSfOff = kSfbOff + kSL * kSfbBytes;     // W4A8: atom of 1.0 scales
  static constexpr int kBarOff = kUnitSfOff + kAtomBytes;
  static constexpr int kNumBars = 3 * kSL + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // MoE: expert offsets [E+1], tile prefix [E+1] and each expert's weight tensor scale [E]
  static constexpr int kMoeOff = kMiscOff + 64;
  static constexpr int kMoeBytes = MOE ? (3 * kMxMoeMaxExperts + 2) * 4 : 0;
  // the epilogue warps' transpose scratch ([warp][8 tokens][32 rows] bf16, 16-byte aligned) where
  // two CTAs per SM still fit with it
  static constexpr int kEpiOff = (kMoeOff + kMoeBytes + 15) / 16 * 16;
  static constexpr int kEpiBytes = 4 * 8 * 32 * 2;
  static constexpr bool kVecEpi = 1024 + kEpiOff + kEpiBytes <= 113 * 1024;
  static constexpr int kSmem = 1024 + (kVecEpi ? kEpiOff + kEpiBytes : kMoeOff + kMoeBytes);
  // TMEM: accumulator [0, BT), then scale-factor slots
  static constexpr int kSfCols = NV ? kSL * 32 : kSL * 4 + 4;
  static constexpr int kColsNeeded = BT + kSfCols;
  static constexpr uint32_t kTmemCols = kColsNeeded <= 32 ? 32 : kColsNeeded <= 64 ? 64 : kColsNeeded <= 128 ? 128
                                        : 256;
  static_assert(kColsNeeded <= 256, "TMEM budget: two CTAs per SM");
  static_assert(kSmem <= 113 * 1024, "shared memory: two CTAs per SM");
  static_assert(kSL >= 2, "pipeline depth");
};

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

// Largest e with prefix[e] <= tile (prefix[0] = 0 <= tile < prefix[E]).
__device__ __forceinline__ int mx_find_expert(const int32_t* prefix, int experts, int tile) {
  int lo = 0, hi = experts;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  return lo;
}

struct MxTile {
  int32_t nt;      // weight tile (128 rows)
  int32_t e;       // expert (0 when dense)
  int32_t blk;     // W4A4: 128-row block of the activation scale atoms
  int64_t m0, m_end;
};

// Dense tile order: m-major (the CTAs of a wave share a token tile and stream different weight
// tiles), or, with group_m > 1, grouped: within a group of group_m token tiles the token tile
// changes fastest, so a wave covers group_m token tiles and ~CTAs / group_m weight tiles, and each
// weight tile is read from DRAM once per group instead of once per wave.
__device__ __forceinline__ void mx_dense_tile(const MxParams& p, int tile, int& mt, int& nt) {
  if (p.group_m > 1) {
    const int per = p.group_m * p.num_n_tiles;
    const int g = tile / per, local = tile - g * per;
    const int left = p.num_m_tiles - g * p.group_m;
    const int rows = left < p.group_m ? left : p.group_m;
    mt = g * p.group_m + local % rows;
    nt = local / rows;
  } else {
    nt = tile % p.num_n_tiles;
    mt = tile / p.num_n_tiles;
  }
}

template <int BT, bool NV, bool MOE>
__device__ __forceinline__ MxTile mx_decode(const MxParams& p, int tile, const int32_t* prefix, const int32_t* offs) {
  MxTile t;
  if (!MOE) {
    int mt;
    mx_dense_tile(p, tile, mt, t.nt);
    t.e = 0;
    t.m0 = static_cast<int64_t>(mt) * BT;
    t.m_end = p.m < t.m0 + BT ? p.m : t.m0 + BT;
    t.blk = static_cast<int32_t>(t.m0 / 128);
  } else {
    t.e = mx_find_expert(prefix, p.num_experts, tile);
    const int local = tile - prefix[t.e];
    t.nt = local % p.num_n_tiles;
    const int mt = local / p.num_n_tiles;
    t.m0 = static_cast<int64_t>(offs[t.e]) + static_cast<int64_t>(mt) * BT;
    t.m_end = offs[t.e + 1] < t.m0 + BT ? offs[t.e + 1] : t.m0 + BT;
    t.blk = prefix[t.e] / p.num_n_tiles + mt;   // token tiles of the experts before, then this one's
  }
  return t;
}

template <int BT, bool NV, bool MOE>
__global__ void __launch_bounds__(threads_of<NV>(), kMxCtasPerSm) mx_gemm_kernel(const __grid_constant__ MxParams p) {
  using S = MxShape<BT, NV, MOE>;
  constexpr int SL = S::kSL;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + SL;
  uint64_t* sf_full = bars + 2 * SL;     // [stage] its scale factors are in TMEM (commit)
  uint64_t* acc_full = sf_full + SL;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + S::kMiscOff + 4);
  float* gw_sh = reinterpret_cast<float*>(smem + S::kMiscOff + 8);
  int32_t* offs = reinterpret_cast<int32_t*>(smem + S::kMoeOff);          // MoE: [E+1]
  int32_t* prefix = offs + (MOE ? kMxMoeMaxExperts + 1 : 0);              // MoE: [E+1]
  float* gw_e = reinterpret_cast<float*>(prefix + (MOE ? kMxMoeMaxExperts + 1 : 0));   // MoE: [E]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (MOE) {
    // The MoE set-up warp may raise the abort flag while thread 0 is still setting up: clear the
    // flag before any role runs, so that a raised flag is never overwritten.
    if (threadIdx.x == 0) *abort_flag = 0u;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < SL; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], NV ? 2 : 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, NV ? 3 : 1);   // the MMA thread's (and W4A4's scale-copy threads') last commits
    fence_barrier_init();
    if (!MOE) *abort_flag = 0u;
    const PackedHeader* h = reinterpret_cast<const PackedHeader*>(p.packed);
    if (!(h->magic == kMagic && static_cast<int32_t>(h->fmt) == p.fmt && h->n == p.n && h->k == p.k)) {
      atomicOr(p.err, kErrHeader);
      *abort_flag = 1u;
    }
    *gw_sh = NV ? h->tensor_scale : 1.0f;   // gX is applied by the epilogue (after its wait)
  }
  if (!NV) {
    // unit activation scales (E8M0 127 = 1.0) for every row
    for (int i = threadIdx.x; i < kAtomBytes / 4; i += threads_of<NV>())
      reinterpret_cast<uint32_t*>(smem + S::kUnitSfOff)[i] = 0x7F7F7F7Fu;
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(tmem_slot, S::kTmemCols);
  if (MOE && warp == 2) {
    // Every expert's header (the weights never depend on the previous kernel, so before its
    // wait), then the offsets (which may): per-expert token tiles x weight tiles, exclusive
    // prefix. Malformed offsets or a header that does not match set the error word and abort.
    const int E = p.num_experts;
    bool bad_hdr = false;
    for (int e = lane; e < E; e += 32) {
      const PackedHeader* h = reinterpret_cast<const PackedHeader*>(p.packed + static_cast<size_t>(e) * p.expert_stride);
      bad_hdr |= !(h->magic == kMagic && static_cast<int32_t>(h->fmt) == p.fmt && h->n == p.n && h->k == p.k);
      gw_e[e] = NV ? h->tensor_scale : 1.0f;
    }
    pdl_wait();
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int local = 0;
    bool bad = false;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const int a = p.offsets[e], b = p.offsets[e + 1];
        bad |= (b < a) || (a < 0) || (b > p.m);
        offs[e] = a;
        local += b > a ? ((b - a + BT - 1) / BT) * p.num_n_tiles : 0;
      }
    }
    if (lane == 0) {
      offs[E] = p.offsets[E];
      bad |= p.offsets[0] != 0;
    }
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        prefix[e] = run;
        const int a = p.offsets[e], b = p.offsets[e + 1];
        run += b > a ? ((b - a + BT - 1) / BT) * p.num_n_tiles : 0;
      }
    }
    if (lane == 31) prefix[E] = incl;
    if (__any_sync(0xffffffffu, bad_hdr) && lane == 0) atomicOr(p.err, kErrHeader);
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, kErrOffsets);
    if (__any_sync(0xffffffffu, bad || bad_hdr) && lane == 0) *abort_flag = 1u;
  }
  __syncthreads();
  if (threadIdx.x == 0) pdl_launch_dependents();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sf_col0 = BT;  // first scale-factor column
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns, true};   // waiting roles suspend (mbar_try_wait_suspend)
  SchedIter sched;
  sched.init(p.sched, MOE ? prefix[p.num_experts] : p.sched.num_tiles, blockIdx.x);
  const int kb_total = p.sched.kb_total;
  const bool aborted_early = *abort_flag != 0u;

  if (aborted_early) {
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tmap_w);
      prefetch_tmap(&p.tmap_x);
      // Weights are streamed once when one token tile covers M; otherwise other CTAs re-read them.
      const bool reuse_w = MOE || p.num_m_tiles > 1;
      const uint64_t pol_w = reuse_w ? policy_evict_last() : policy_evict_first();
      const uint64_t pol_x = reuse_w ? policy_evict_normal() : policy_evict_last();
      // The W4A8 weight load reads 8 KB of packed codes and spreads them over 16 KB of shared
      // memory (16U4_ALIGN16B); its transaction count is the 8 KB read.
      const uint32_t w_tx = static_cast<uint32_t>((NV ? kWTile : kWTile / 2) + S::kSfaBytes);
      const uint32_t x_tx = static_cast<uint32_t>(S::kXStage + S::kSfbBytes);
      auto load_w = [&](int slot, int nt, int e, int kb) {
        if (MOE)
          tma_3d_g2s(smem + S::kWOff + slot * kWTile, &p.tmap_w, kb * 128, nt * 128, e, &full[slot], pol_w);
        else
          tma_2d_g2s(smem + S::kWOff + slot * kWTile, &p.tmap_w, kb * 128, nt * 128, &full[slot], pol_w);
        const size_t atom = NV ? static_cast<size_t>(nt) * (kb_total * 4) + static_cast<size_t>(kb) * 4
                               : static_cast<size_t>(nt) * kb_total + kb;
        const uint8_t* atoms = MOE ? p.w_atoms + static_cast<size_t>(e) * p.expert_stride : p.w_atoms;
        bulk_g2s(smem + S::kSfaOff + slot * S::kSfaBytes, atoms + atom * kAtomBytes, S::kSfaBytes, &full[slot],
                 pol_w);
      };
      int ls = 0;
      uint32_t ph = 0;
      int issued = 0;
      Segment seg;
      bool ok = true;
      // Weights and their scales do not depend on the previous kernel: start streaming the first
      // pipeline stages before waiting for it. Their bytes are announced with expect_tx (no
      // arrive), so a stage cannot complete before its activation part is issued below.
      int pre = 0;
      if (!MOE) {   // (the MoE tile list needs the offsets, which may come from the previous kernel)
        SchedIter pf = sched;
        Segment ps;
        while (pre < SL && pf.next(ps)) {
          int mt, nt;
          mx_dense_tile(p, ps.tile, mt, nt);
          for (int kb = ps.kb0; kb < ps.kb1 && pre < SL; ++kb, ++pre) {
            mbar_expect_tx(&full[pre], w_tx);
            load_w(pre, nt, 0, kb);
          }
        }
      }
      pdl_wait();
      while (ok && sched.next(seg)) {
        const MxTile t = mx_decode<BT, NV, MOE>(p, seg.tile, prefix, offs);
        const int m0 = static_cast<int>(t.m0);
        for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
          if (issued >= pre) {
            if (!mbar_wait(&empty[ls], ph ^ 1u, wc)) { ok = false; break; }
            mbar_expect_tx(&full[ls], w_tx);
            load_w(ls, t.nt, t.e, kb);
          }
          mbar_arrive_expect_tx(&full[ls], x_tx);
          tma_2d_g2s(smem + S::kXOff + ls * S::kXStage, &p.tmap_x, kb * 128, m0, &full[ls], pol_x);
          if (NV) {
            bulk_g2s(smem + S::kSfbOff + ls * S::kSfbBytes,
                     p.x_atoms + (static_cast<size_t>(t.blk) * (p.k / 64) + static_cast<size_t>(kb) * 4) * kAtomBytes,
                     S::kSfbBytes, &full[ls], pol_x);
          }
          ++issued;
          if (++ls == SL) { ls = 0; ph ^= 1u; }
        }
      }
      if (*abort_flag) {
        const int n = issued < SL ? issued : SL;
        for (int i = 0; i < n; ++i) {
          if (--ls < 0) { ls = SL - 1; ph ^= 1u; }
          drain_wait(&full[ls], ph, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per k-block: wait for the stage (W4A4: until its scale factors are in TMEM, which implies
    // its operands have landed), copy its weight scales (W4A8), then its MMAs. W4A4's eight scale
    // copies per block run on their own warp: a thread that issues tcgen05 work stalls at its
    // next shared-memory access until that work is under way, so they would otherwise lengthen
    // every k-block of this thread.
    if (lane == 0) {
      const uint32_t unit_sfb = tmem + sf_col0 + (NV ? 0 : SL * 4);
      if (!NV) tc_cp_32x128b_x4(unit_sfb, sdesc_sf(smem_u32(smem + S::kUnitSfOff)));
      int ls = 0;
      uint32_t ph = 0, acc_i = 0;
      Segment seg;
      bool ok = true;
      while (ok && sched.next(seg)) {
        if (!mbar_wait(acc_empty, (acc_i & 1u) ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem;
        for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
          if (!mbar_wait(NV ? &sf_full[ls] : &full[ls], ph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t w_base = smem_u32(smem + S::kWOff + ls * kWTile);
          const uint32_t x_base = smem_u32(smem + S::kXOff + ls * S::kXStage);
          if (NV) {
            const uint32_t slot = tmem + sf_col0 + ls * 32;
            constexpr uint32_t idesc = idesc_block_scaled(128, BT, 1, 1, 0, 0, 0);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = sdesc_sw128(w_base + k * 32);
              const uint64_t bd = sdesc_sw128(x_base + k * 32);
              mma_mxf4nvf4_4x(d, ad, bd, idesc, slot + 4 * k, slot + 16 + 4 * k, (kb > seg.kb0 || k > 0) ? 1u : 0u);
            }
          } else {
            const uint32_t slot = tmem + sf_col0 + ls * 4;
            tc_cp_32x128b_x4(slot, sdesc_sf(smem_u32(smem + S::kSfaOff + ls * S::kSfaBytes)));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t idesc = idesc_block_scaled(128, BT, 5, 0, 1, k, k);
              const uint64_t ad = sdesc_sw128(w_base + k * 32);
              const uint64_t bd = sdesc_sw128(x_base + k * 32);
              mma_mxf8f6f4(d, ad, bd, idesc, slot, unit_sfb, (kb > seg.kb0 || k > 0) ? 1u : 0u);
            }
          }
          tc_commit(&empty[ls]);
          if (++ls == SL) { ls = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(acc_full);
        ++acc_i;
      }
      tc_commit(drain);
      drain_wait(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (NV && (warp == kSfWarp || warp == kSfWarp + 1)) {
    // ------------------------------------------------------------ scale-factor copies
    // For every k-block in order: once the stage has landed, copy its scale atoms from shared
    // memory to the stage's TMEM slot (tcgen05.cp.32x128b.warpx4 puts row r's four scales in lane
    // r%32 of column r/32 of a 4-column slot) and commit to sf_full. A slot is rewritten only
    // after the producer refilled its stage, i.e. after the MMAs that read it completed.
    if (lane == 0) {
      const bool act = warp == kSfWarp + 1;   // warp 6: weight scales, warp 7: activation scales
      int ls = 0;
      uint32_t ph = 0;
      Segment seg;
      bool ok = true;
      while (ok && sched.next(seg)) {
        for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
          if (!mbar_wait(&full[ls], ph, wc)) { ok = false; break; }
          const uint32_t src = act ? smem_u32(smem + S::kSfbOff + ls * S::kSfbBytes)
                                   : smem_u32(smem + S::kSfaOff + ls * S::kSfaBytes);
          const uint32_t slot = tmem + sf_col0 + ls * 32 + (act ? 16 : 0);
#pragma unroll
          for (int j = 0; j < 4; ++j) tc_cp_32x128b_x4(slot + 4 * j, sdesc_sf(src + j * kAtomBytes));
          tc_commit(&sf_full[ls]);
          if (++ls == SL) { ls = 0; ph ^= 1u; }
        }
      }
      tc_commit(drain);
      drain_wait(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ epilogue warps (2..5)
    pdl_wait();   // Y, s_tok, partials and counters: wait for the previous kernel
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const int64_t total_it = static_cast<int64_t>(p.sched.num_tiles) * kb_total;
    const float gscale = NV ? *gw_sh * (*p.x_global) : 1.0f;
    // 16-byte stores of Y through the transpose scratch (Y 16-byte aligned, N % 8 == 0)
    const bool vec_y = S::kVecEpi && (reinterpret_cast<uintptr_t>(p.y) & 15u) == 0 && (p.n & 7) == 0;
    uint32_t acc_i = 0;
    bool first_seg = true;
    Segment seg;
    while (sched.next(seg)) {
      const MxTile t = mx_decode<BT, NV, MOE>(p, seg.tile, prefix, offs);
      const float gs = MOE && NV ? gw_e[t.e] * (*p.x_global) : gscale;
      if (!mbar_wait(acc_full, acc_i & 1u, wc)) break;
      tc_fence_after();
      const int64_t m0 = t.m0;
      const int64_t m_end = t.m_end;
      const int64_t n = static_cast<int64_t>(t.nt) * 128 + row;
      const bool full_seg = seg.kb0 == 0 && seg.kb1 == kb_total;
      // Stream-K tile shared by CTAs c_lo .. c_hi: the owner (holding k-block 0) waits for the
      // others' published partials and adds them to its own accumulator; the others publish.
      const bool owner = !full_seg && seg.kb0 == 0;
      uint32_t* flag = full_seg ? nullptr
                                : sk_flag(p.counters, owner ? blockIdx.x
                                                            : sk_tile_owner(seg.tile, kb_total, total_it, p.sched.grid), q);
      int64_t c_hi = 0;
      bool have = true;
      if (owner) {
        c_hi = sk_owner(static_cast<int64_t>(seg.tile + 1) * kb_total - 1, total_it, p.sched.grid);
        have = sk_wait(flag, static_cast<uint32_t>(c_hi - blockIdx.x), wc);
      }
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16);
      float* slotp = p.partial + (static_cast<size_t>(blockIdx.x) * 2 + (first_seg ? 0 : 1)) * BT * 128 +
                     static_cast<size_t>(row) * BT;
#pragma unroll 1
      for (int j0 = 0; j0 < BT && have; j0 += 16) {
        uint32_t v[16];
        tmem_ld16(tbase + j0, v);
        tmem_wait_ld();
        if (full_seg || owner) {
          float a[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) a[jj] = __uint_as_float(v[jj]);
          if (owner)
            sk_add_partials<BT>(p.partial, total_it, p.sched.grid, kb_total, seg.tile, blockIdx.x, c_hi, row, j0, a);
          if (vec_y) {
            // Transpose 8 tokens at a time through shared memory, so that each store moves 8
            // consecutive rows (16 bytes) of one token.
            const uint32_t sc8 = smem_u32(smem + S::kEpiOff) + static_cast<uint32_t>(q) * (8 * 32 * 2);
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int64_t m = m0 + j0 + 8 * h8 + jj;
                const float scl = m < m_end ? (NV ? gs : p.s_tok[m]) : 0.f;
                const uint16_t hb = __bfloat16_as_ushort(__float2bfloat16_rn(a[8 * h8 + jj] * scl));
                asm volatile("st.shared.u16 [%0], %1;" ::"r"(sc8 + (jj * 32 + lane) * 2), "h"(hb) : "memory");
              }
              __syncwarp();
              const int tt = lane >> 2, c8 = lane & 3;   // token, 8-row group
              const uint4 v8 = ld_shared_v4(sc8 + (tt * 32 + 8 * c8) * 2);
              const int64_t m = m0 + j0 + 8 * h8 + tt;
              const int64_t n8 = static_cast<int64_t>(t.nt) * 128 + 32 * q + 8 * c8;
              if (m < m_end) {
                if (n8 + 8 <= p.n) {
                  *reinterpret_cast<uint4*>(p.y + m * p.n + n8) = v8;
                } else {
                  const uint32_t w4[4] = {v8.x, v8.y, v8.z, v8.w};
                  for (int e = 0; e < 8 && n8 + e < p.n; ++e)
                    p.y[m * p.n + n8 + e] = __ushort_as_bfloat16(static_cast<uint16_t>(w4[e >> 1] >> (16 * (e & 1))));
                }
              }
              __syncwarp();   // the scratch is rewritten by the next 8 tokens
            }
          } else if (n < p.n) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int64_t m = m0 + j0 + jj;
              if (m < m_end) {
                const float sc = NV ? gs : p.s_tok[m];
                p.y[m * p.n + n] = __float2bfloat16_rn(a[jj] * sc);
              }
            }
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(slotp + j0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      ++acc_i;
      if (!full_seg && !owner) sk_publish(flag, lane);
      if (owner && have) {
        __syncwarp();
        if (lane == 0) *flag = 0u;
      }
      first_seg = false;
    }
  }

  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::kTmemCols);
  }
}

template <int BT, bool NV, bool MOE>
cudaError_t launch_one(const MxParams& p, cudaStream_t st) {
  using S = MxShape<BT, NV, MOE>;
  auto kern = mx_gemm_kernel<BT, NV, MOE>;
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return launch_pdl(kern, p.sched.grid, threads_of<NV>(), S::kSmem, st, p);
}

template <bool NV, bool MOE>
cudaError_t launch_bt(const MxParams& p, int tile_m, cudaStream_t st) {
  switch (tile_m) {
    case 16: return launch_one<16, NV, MOE>(p, st);
    case 32: return launch_one<32, NV, MOE>(p, st);
    case 64: return launch_one<64, NV, MOE>(p, st);
    case 128: return launch_one<128, NV, MOE>(p, st);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace
}  // namespace hm
