// W4A16 GEMM for decode-sized M (up to 32 tokens): Y[M,N] = X[M,K] * dequant(W)^T, with
// warp-level bf16 MMA (mma.sync m16n8k16, fp32 accumulation) as the multiply engine.
//
// Same product and restore rule as the tcgen05 W4A16 kernels (the explainer page "vLLM
// Humming은 4비트를 어떻게 계산하나", sections "4비트 값에는 스케일이라는 해석 규칙이 붙는다" and
// "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다"). With at most 32 tokens every weight byte
// feeds at most 64 multiply-adds: the product is bound by streaming the packed weights from HBM,
// and what limits a kernel is the work per weight on the SM (dequant, operand staging, hand-offs
// between roles), not MMA throughput. The tcgen05 path spends that on restoring weights into
// TMEM, single-thread MMA issue and accumulator hand-offs per 128-K block; here each warp restores
// its weights in registers straight into the MMA's A fragment and keeps its accumulators in
// registers, so the only hand-off per unit is the shared-memory stage itself.
//
//  * Work: the packed 128x128 units (n-tile major: unit u is tile u / kb, k-block u % kb) are cut
//    into one contiguous range per CTA, start(c) = floor(c * U / G). The planner takes G = tiles x
//    floor(SMs / tiles) when tiles <= SMs (every CTA then holds one K range of one tile), else
//    G = SMs (a range may cover the tail of one tile, whole tiles and the head of another).
//  * Roles (persistent CTA per SM): a producer warp loads each unit with a bulk copy (the first
//    stages from one lane each) and the activation block X[0:MT, k-block] with one 2-D TMA load
//    (token rows past M read as zeros) into a ring of stages; consumer warp (p, c, r) takes rows
//    32p..32p+31 (two 16-row MMA tiles) and the 32-K chunks 2c, 2c+1 of the units of parity r: for
//    up to 16 tokens two parities take alternate units (16 consumer warps, four per SM
//    sub-partition, hiding each other's load and MMA latencies), for 32 tokens one parity (8 warps,
//    each holding four token groups of sums). An INT4 metadata warp turns each unit's 128 scales
//    and zero-points into fp32 scales and bf16x2 (128 + z) pairs once. The walk over units, slots
//    and phases advances by counting (no division per unit).
//  * Fragments: for m16n8k16, lane (g = lane/4, t = lane%4) holds A pairs at MMA k-slots
//    {2t, 2t+1} and {2t+8, 2t+9}, B pairs at the same slots for token g. A contraction may number
//    its k in any order as long as A and B agree, so lane t takes the 32-bit code word t of its
//    rows (8 consecutive k) and the 8 matching activations: one 32-bit load per weight row, one
//    16-byte load of activations per 8 tokens, no shuffles. Two MMAs per word (k-slots 0-7 from
//    the word's columns 0-3, then columns 4-7).
//  * INT4: the word is restored to exact bf16 (u - z) pairs (one shift, one lop3, one bf16x2
//    subtract per pair); each unit's MMAs accumulate sum (u - z) x over the unit's 128 K in fp32,
//    and the group scale multiplies that sum (s * sum (u - z) x, as in the small-token tcgen05
//    kernel). MXFP4 and MXINT4: the word is restored with its E8M0 scale (exact; MXINT4 through
//    the INT4 restore with z = 8 and a bf16 power-of-two scale) and the MMAs accumulate
//    straight into the running sums.
//  * Segment end: the warps of a row pair (two or four) add their sums in a fixed order through shared
//    memory (mbarrier hand-off, bounded); every warp closes every segment of its CTA's range, even
//    one that holds no unit of its parity. A tile owned whole by the CTA is written to Y. A tile
//    shared by several CTAs has a fixed owner, the CTA holding its first k-block: it reaches the
//    tile at the end of its range, while for every other contributor the tile is the first
//    segment. Those store fp32 partials ([CTA][token][row]) and add 1 to a per-(tile, row pair)
//    counter with a release (no waiting); the owner waits (bounded, acquire) for the count, adds
//    the partials in CTA order to its own (deterministic), writes Y and clears the counter.
//    When every tile is cut into 2-4 K ranges, one per CTA, the ranges of a tile form a thread-block
//    cluster instead: ranks 1.. store their sums straight into rank 0's shared memory and arrive on
//    its barrier (release at cluster scope), rank 0 waits (bounded) and adds them in rank order,
//    the same order as the global path, so both give identical bits. A cluster barrier after set-up
//    and one before exit keep every remote access inside the lifetime of the CTA it targets; the
//    launcher uses clusters only when the device can hold all of them at once.
//  * Every mbarrier wait is bounded (device error word + CTA abort flag); the producer drains its
//    copies in flight before the CTA exits; PDL as in the other kernels (weights are loaded before
//    griddepcontrol.wait, activations and outputs only after it).
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

// Warps: 0 producer, then the consumers, then the INT4 row-metadata warp. Consumer warp (row pair,
// chunk pair, unit parity): 4 x 2 x kPar. Up to 16 tokens two parities take alternate units (16
// consumers, four per sub-partition, to hide load and MMA latency); with 32 tokens a warp holds four
// token groups of sums and there is one parity (8 consumers, twice the registers each).
constexpr int kVCons0 = 1;
__host__ __device__ constexpr int v_par(int mt) { return mt <= 16 ? 2 : 1; }
__host__ __device__ constexpr int v_consumers(int mt) { return 8 * v_par(mt); }
__host__ __device__ constexpr int v_meta_warp(int mt) { return kVCons0 + v_consumers(mt); }
__host__ __device__ constexpr int v_threads(int mt) { return 32 * (v_meta_warp(mt) + 1); }

template <int MT, int WB = 8704, bool MOE = false>
struct VShape {
  static constexpr int kNQ = MT / 8;                // token groups of 8 (MMA N)
  static constexpr int kWBytes = WB;                // one unit (the largest of the formats served)
  // activations: MT token rows of 128 bf16, as one TMA box lands them. The two token rows a
  // quarter-warp reads then share banks (a 2-way conflict on two loads per warp and unit), which
  // costs less than a wider, padded box: the activation box is a TMA operation per unit, and a
  // 160-column box with a 320-byte pitch made the load pipeline ~25 % slower (measured)
  static constexpr int kXPitch = 256;
  static constexpr int kXBytes = MT * kXPitch;
  // INT4 row metadata of the unit, written by the metadata warp: [128 rows] {fp32 scale, bf16x2
  // (128 + z, 128 + z)}
  static constexpr int kMetaOff = kWBytes + kXBytes;
  static constexpr int kStage = kMetaOff + 128 * 8;
  static constexpr int kPar = v_par(MT);
  // segment-end exchange: [row pair][the 2 kPar - 1 other warps][lane][2 tiles x 4 x kNQ floats]
  static constexpr int kXchgFloats = 8 * kNQ;
  static constexpr int kXchgBytes = 4 * (2 * kPar - 1) * 32 * kXchgFloats * 4;
  // cluster hand-off of a shared tile: [rank 1..3][row pair][lane][2 tiles x 4 x kNQ floats] in
  // the owner CTA (rank 0)
  static constexpr int kRedBytes = MOE ? 0 : 3 * 4 * 32 * kXchgFloats * 4;   // (no clusters when grouped)
  // as many stages (even, at most 16) as the 227 KB per CTA leave beside the fixed parts
  // grouped (MoE) variant: expert offsets [E+1] and token-tile prefix [E+1]
  static constexpr int kMoeBytes = MOE ? 2 * (kGemvMoeMaxExperts + 1) * 4 : 0;
  static constexpr int kFixed = kXchgBytes + kRedBytes + (3 * 16 + 3 * 4) * 8 + 64 + 16 * 4 + 128 + kMoeBytes;
  static constexpr int kSFit = (232448 - kFixed) / kStage;
  static constexpr int kS = (kSFit > 16 ? 16 : kSFit) & ~1;
  static_assert(kS % kPar == 0, "a stage always holds units of one parity");
  static constexpr int kXchgOff = kS * kStage;
  static constexpr int kRedOff = kXchgOff + kXchgBytes;
  static constexpr int kBarOff = kRedOff + kRedBytes;
  static constexpr int kNumBars = 3 * kS + 3 * 4;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kMoeOff = kMiscOff + 64 + 16 * 4;
  static constexpr int kSmem = kMoeOff + kMoeBytes + 128;   // + e2m1 table, MoE arrays, alignment slack
  static_assert(kS >= 4, "pipeline depth");
  static_assert(kWBytes % 128 == 0 && kStage % 128 == 0, "TMA destinations 128-byte aligned");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

constexpr int kVMaxCluster = 4;   // CTAs per cluster for the shared-memory hand-off (ranks 1..3 publish)

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with a zero accumulator (the first MMA of a chain).
__device__ __forceinline__ void mma_bf16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Unit bytes a stage holds for a weight format (WK).
__host__ __device__ constexpr int v_wbytes(int wk) { return wk == 8 ? 16768 : (wk == 6 ? 9472 : 8704); }

// WK: 0 = INT4, 2 = MXFP4, 3 = MXINT4 (the last two carry E8M0 scales per 32 in their units),
// 6 = INT4 with a bf16 scale (and zero-point) per 32-K chunk, applied to each chunk's sum;
// 8 = INT8 (one byte per code, bf16 scale and u8 zero-point per row and 128-K block), restored to the
// exact integers u - z and scaled after the block's sum like INT4.
// MOE: the grouped variant over expert-sorted rows (token tiles of MT rows per expert).
template <int MT, int WK, bool MOE>
__global__ void __launch_bounds__(v_threads(MT), 1) gemv_kernel(const __grid_constant__ F16Params p) {
  using S = VShape<MT, v_wbytes(WK), MOE>;
  constexpr bool MX = WK == 2 || WK == 3;
  constexpr bool G32 = WK == 6;
  constexpr int SL = S::kS;
  constexpr int NQ = S::kNQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);   // unit + activations landed
  uint64_t* empty = full + SL;                                        // stage consumed (8 warps)
  uint64_t* meta_full = empty + SL;                                   // INT4 row metadata written
  uint64_t* xfull = meta_full + SL;                                   // [row pair] 3 warps stored
  uint64_t* xfree = xfull + 4;                                        // [row pair] the 4th read them
  uint64_t* red_full = xfree + 4;                                     // [row pair] cluster ranks 1.. stored
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + S::kMiscOff);
  volatile uint32_t* hz_sh = abort_flag + 1;
  float* lut = reinterpret_cast<float*>(smem + S::kMiscOff + 64);
  float* xchg = reinterpret_cast<float*>(smem + S::kXchgOff);
  float* red = reinterpret_cast<float*>(smem + S::kRedOff);
  int32_t* mtpre = reinterpret_cast<int32_t*>(smem + S::kMoeOff);      // MoE: tile prefix [E+1]
  int32_t* moffs = mtpre + kGemvMoeMaxExperts + 1;                      // MoE: expert offsets [E+1]
  const int csize = (!MOE && p.cluster > 1) ? p.cluster : 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int32_t kb_total = p.sched.kb_total;
  const int m_rows = static_cast<int>(p.m);

  if (MOE) {
    // The MoE set-up warp may raise the abort flag while thread 0 is still setting up: clear the
    // flag before any role runs, so that a raised flag is never overwritten.
    if (threadIdx.x == 0) *abort_flag = 0u;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    trace_mark(p.trace, 0);
    if (p.trace != nullptr) {
      uint32_t smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      p.trace[blockIdx.x * 16 + 13] = smid;
    }
    for (int s = 0; s < SL; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);   // the 8 consumer warps of the stage's unit parity
      mbar_init(&meta_full[s], 1);
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(&xfull[q], 2 * S::kPar - 1);
      mbar_init(&xfree[q], 1);
      mbar_init(&red_full[q], csize > 1 ? csize - 1 : 1);
    }
    fence_barrier_init();
    // (MoE: the expert pointers may come from the previous kernel; the first expert's header
    // decides whether the units carry zero-points, and the set-up warp checks every expert's
    // header against it)
    if (MOE) pdl_wait();
    const uint8_t* first_w = (MOE && p.packed_list != nullptr) ? p.packed_list[0] : p.packed;
    const PackedHeader hdr = *reinterpret_cast<const PackedHeader*>(first_w);
    if (!MOE) *abort_flag = 0u;
    *hz_sh = hdr.has_zero == 1u ? 1u : 0u;
    if (!(hdr.magic == kMagic && static_cast<int32_t>(hdr.fmt) == p.fmt && hdr.n == p.n && hdr.k == p.k)) {
      atomicOr(p.err, kErrHeader);
      *abort_flag = 1u;
    }
  }
  if (WK == 2 && threadIdx.x < 16) lut[threadIdx.x] = e2m1_value(threadIdx.x);
  if (MOE && warp == v_meta_warp(MT)) {
    // Every expert's header against the call and the first expert's zero-point flag (strided
    // weights before the wait for the previous kernel: they never depend on it; a pointer list
    // after it), then the expert offsets (which the previous kernel may write) -> token tiles of
    // MT rows per expert x weight tiles, exclusive prefix over the experts. A header that does not
    // match or malformed offsets set the error word and abort every CTA before any weight is read.
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
  // this CTA's range of the (tile, k-block) space (MoE: the tile count comes from the offsets)
  // (MoE: the launch has one CTA per SM whatever the offsets; with fewer units than CTAs only the
  // first `total` CTAs take one each, so that every CTA between a shared tile's owner and its last
  // contributor holds a part of it, which the owner's arrival count relies on)
  const int64_t total = static_cast<int64_t>(MOE ? mtpre[p.num_experts] : p.sched.num_tiles) * kb_total;
  const int32_t grid = MOE ? static_cast<int32_t>(total < p.sched.grid ? total : p.sched.grid) : p.sched.grid;
  const bool idle = static_cast<int32_t>(blockIdx.x) >= grid;
  const int32_t u0 = idle ? 0 : static_cast<int32_t>(sk_start(blockIdx.x, total, grid));
  const int32_t u1 = idle ? 0 : static_cast<int32_t>(sk_start(blockIdx.x + 1, total, grid));
  const int32_t n_units = u1 - u0;
  const int32_t tile0 = u0 / kb_total, kb0 = u0 - tile0 * kb_total;
  // Cluster barrier, two phases, each split into an arrive and a wait per thread: phase 1 makes the
  // owner's barriers initialised before another CTA of its cluster arrives on them (every thread
  // arrives here, a publishing warp waits just before its first remote access, the others at
  // exit); phase 2 keeps every CTA alive until no other one may still write into its shared
  // memory (a thread arrives once it has no remote access left: a publisher after its stores, the
  // owner's readers once the publications they wait for have landed, the other roles at exit).
  bool cl_waited1 = false, cl_arrived2 = false;
  if (csize > 1) cluster_arrive();
  if (threadIdx.x == 0) {
    pdl_launch_dependents();
    trace_mark(p.trace, 1);
  }
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  const bool aborted_early = *abort_flag != 0u;
  const uint32_t has_zero = *hz_sh;
  const uint32_t kUnit = WK == 8 ? (has_zero ? kUnitInt8Zp : kUnitInt8)
                         : (MX ? kUnitMx : (G32 ? (has_zero ? kUnitG32Zp : kUnitG32) : (has_zero ? kUnitInt4Zp : kUnitInt4)));

  if (aborted_early) {
    // header mismatch: nothing was issued
  } else if (warp == 0) {
    // ---------------------------------------------------------------- producer
    const uint64_t pol_w = policy_evict_first();
    const uint8_t* wsrc = p.packed + kHeaderBytes + static_cast<size_t>(u0) * kUnit;
    const uint32_t stage_bytes = kUnit + static_cast<uint32_t>(S::kXBytes);
    const int first = n_units < SL ? n_units : SL;
    if constexpr (MOE) {
      // Grouped: unit i of the range is k-block (kb0 + i) % kb of tile tile0 + (kb0 + i) / kb, whose
      // expert, weight tile and first token row come from the prefix (token rows of the box past the
      // expert's end belong to the next expert or read as zeros; their sums are never stored). Every
      // header was checked in the set-up. The first stages one per lane, then lane 0.
      const uint64_t pol_x = policy_evict_last();
      if (lane == 0) prefetch_tmap(&p.tmap_x);
      if (lane < first) {
        const int kb_l = (kb0 + lane) % kb_total;
        const TileInfo t0 = decode_tile<MT, true>(p, tile0 + (kb0 + lane) / kb_total, mtpre, moffs, kUnit);
        mbar_arrive_expect_tx(&full[lane], stage_bytes);
        bulk_g2s(smem + lane * S::kStage, t0.wbase + static_cast<size_t>(kb_l) * kUnit, kUnit, &full[lane], pol_w);
        tma_2d_g2s(smem + lane * S::kStage + S::kWBytes, &p.tmap_x, kb_l * 128, t0.m0, &full[lane], pol_x);
      }
      __syncwarp();
      if (lane == 0) {
        int issued = first;
        if (first < n_units) {
          int32_t tl = tile0 + (kb0 + first) / kb_total;
          int kb = (kb0 + first) % kb_total;
          TileInfo t = decode_tile<MT, true>(p, tl, mtpre, moffs, kUnit);
          int s = 0;
          uint32_t ph = 0;
          for (int i = first; i < n_units; ++i) {
            if (!mbar_wait(&empty[s], ph, wc)) break;
            mbar_arrive_expect_tx(&full[s], stage_bytes);
            bulk_g2s(smem + s * S::kStage, t.wbase + static_cast<size_t>(kb) * kUnit, kUnit, &full[s], pol_w);
            tma_2d_g2s(smem + s * S::kStage + S::kWBytes, &p.tmap_x, kb * 128, t.m0, &full[s], pol_x);
            issued = i + 1;
            if (++kb == kb_total && issued < n_units) {
              kb = 0;
              t = decode_tile<MT, true>(p, ++tl, mtpre, moffs, kUnit);
            }
            if (++s == SL) { s = 0; ph ^= 1u; }
          }
        }
        trace_mark(p.trace, 3);
        // nothing may still be landing in shared memory when the CTA exits
        for (int i = issued - SL < 0 ? 0 : issued - SL; i < issued; ++i)
          drain_wait(&full[i % SL], static_cast<uint32_t>(i / SL) & 1u, p.timeout_ns);
      }
    } else {
      // Start-up, one stage per lane (a single thread takes ~70 ns per bulk-copy issue): the weights
      // of the first few stages before waiting for the previous kernel (weights are never written
      // by another kernel), then, after the wait, their activation blocks, and only then the rest of
      // the first stages, weights and activations. The TMA unit works through its copies roughly in
      // issue order, so the first stages complete without queueing behind the whole ring's weights.
      constexpr int kEarly = 4;
      const int early = first < kEarly ? first : kEarly;
      if (lane < early) {
        mbar_arrive_expect_tx(&full[lane], stage_bytes);
        bulk_g2s(smem + lane * S::kStage, wsrc + static_cast<size_t>(lane) * kUnit, kUnit, &full[lane], pol_w);
      }
      if (lane == 0) {
        trace_mark(p.trace, 2);
        prefetch_tmap(&p.tmap_x);
      }
      const uint64_t pol_x = policy_evict_last();
      pdl_wait();
      if (lane == 0) trace_mark(p.trace, 5);
      const int kb_lane = (kb0 + lane) % kb_total;   // k-block of stage `lane`
      if (lane < early) tma_2d_g2s(smem + lane * S::kStage + S::kWBytes, &p.tmap_x, kb_lane * 128, 0, &full[lane], pol_x);
      __syncwarp();
      if (lane >= early && lane < first) {
        mbar_arrive_expect_tx(&full[lane], stage_bytes);
        bulk_g2s(smem + lane * S::kStage, wsrc + static_cast<size_t>(lane) * kUnit, kUnit, &full[lane], pol_w);
        tma_2d_g2s(smem + lane * S::kStage + S::kWBytes, &p.tmap_x, kb_lane * 128, 0, &full[lane], pol_x);
      }
      __syncwarp();
      if (lane == 0) {
        int kb = (kb0 + first) % kb_total;
        int issued = first, s = 0;
        uint32_t ph = 0;
        for (int i = first; i < n_units; ++i) {
          if (!mbar_wait(&empty[s], ph, wc)) break;
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          bulk_g2s(smem + s * S::kStage, wsrc + static_cast<size_t>(i) * kUnit, kUnit, &full[s], pol_w);
          tma_2d_g2s(smem + s * S::kStage + S::kWBytes, &p.tmap_x, kb * 128, 0, &full[s], pol_x);
          if (++kb == kb_total) kb = 0;
          issued = i + 1;
          if (++s == SL) { s = 0; ph ^= 1u; }
        }
        trace_mark(p.trace, 3);
        // nothing may still be landing in shared memory when the CTA exits
        for (int i = issued - SL < 0 ? 0 : issued - SL; i < issued; ++i)
          drain_wait(&full[i % SL], static_cast<uint32_t>(i / SL) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == v_meta_warp(MT)) {
    // ---------------------------------------------------------------- INT4 row metadata
    // Each unit's 128 scales and zero-points, once per unit instead of once per consumer warp:
    // lane l converts rows 4l .. 4l+3 (bf16 scale -> fp32, u4 zero-point -> bf16x2 128 + z).
    if constexpr (WK == 8) {
      // INT8: per row {fp32 scale, fp32 2^23 + z} (z = 128 without zero-points: codes are q + 128)
      const uint32_t smem0 = smem_u32(smem);
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < n_units; ++i) {
        if (!mbar_wait(&full[s], ph, wc)) break;
        const uint32_t base = smem0 + s * S::kStage;
        uint32_t sc01, sc23, z4 = 0x80808080u;
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(sc01), "=r"(sc23) : "r"(base + kUnitInt8Codes + 8 * lane));
        if (has_zero) z4 = lds32(base + kUnitInt8 + 4 * lane);
        float zf[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) zf[r] = 8388608.0f + static_cast<float>((z4 >> (8 * r)) & 0xFFu);
        const uint32_t mb = base + S::kMetaOff + 32 * lane;
        st_shared_v4(mb, sc01 << 16, __float_as_uint(zf[0]), sc01 & 0xFFFF0000u, __float_as_uint(zf[1]));
        st_shared_v4(mb + 16, sc23 << 16, __float_as_uint(zf[2]), sc23 & 0xFFFF0000u, __float_as_uint(zf[3]));
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta_full[s]);
        if (++s == SL) { s = 0; ph ^= 1u; }
      }
    } else if constexpr (WK == 0) {
      const uint32_t smem0 = smem_u32(smem);
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < n_units; ++i) {
        if (!mbar_wait(&full[s], ph, wc)) break;
        const uint32_t base = smem0 + s * S::kStage;
        uint32_t sc01, sc23, zz = 0x8888u;
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(sc01), "=r"(sc23) : "r"(base + kUnitCodes + 8 * lane));
        if (has_zero) {
          uint16_t zb;
          asm volatile("ld.shared.u16 %0, [%1];" : "=h"(zb) : "r"(base + kUnitInt4 + 2 * lane));
          zz = zb;
        }
        uint32_t z2[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const uint32_t z = (zz >> (4 * r)) & 0xFu;
          z2[r] = (0x43004300u | z) | (z << 16);
        }
        const uint32_t mb = base + S::kMetaOff + 32 * lane;
        st_shared_v4(mb, sc01 << 16, z2[0], sc01 & 0xFFFF0000u, z2[1]);
        st_shared_v4(mb + 16, sc23 << 16, z2[2], sc23 & 0xFFFF0000u, z2[3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta_full[s]);
        if (++s == SL) { s = 0; ph ^= 1u; }
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int cw = warp - kVCons0;
    const int par = cw >> 3;                 // units u0 + par, u0 + par + kPar, ...
    const int pr = (cw >> 1) & 3;            // row pair: rows 32pr .. 32pr + 31
    const int cp = cw & 1;                   // 32-K chunks 2cp and 2cp + 1 of every unit
    const int slot_id = cp + 2 * par;        // 0 reads the others of its row pair at a segment end
    const int g = lane >> 2, t = lane & 3;
    // fragment rows: tile j (0, 1) of the pair, rows g and g + 8 of the tile
    int rows[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      rows[j][0] = 32 * pr + 16 * j + g;
      rows[j][1] = rows[j][0] + 8;
    }
    // shared-memory offsets within a stage (the per-(tile, row, chunk) parts are immediates):
    // code word t of row 32pr + g (+16j, +8hl) in chunk 2cp (+cc); activation fragment of token g
    // (+8q), columns 64cp + 8t (+32cc); the row's metadata (INT4) or E8M0 scale word (MXFP4, MXINT4)
    const uint32_t woff = static_cast<uint32_t>((2 * cp) * 2048 + (32 * pr + g) * 16 + 4 * t);
    const uint32_t xoff = static_cast<uint32_t>(S::kWBytes + g * S::kXPitch + (2 * cp) * 64 + t * 16);
    const uint32_t moff = static_cast<uint32_t>(MX ? kUnitCodes + (32 * pr + g) * 4 : S::kMetaOff + (32 * pr + g) * 8);
    const uint32_t smem0 = smem_u32(smem);

    float yacc[2][NQ][4];   // [tile][token group][c0..c3]: rows g / g+8 x tokens 2t, 2t+1
    int seg_kb0 = kb0, seg_count = 0;

    // The segment [seg_kb0, seg_kb1) of `tile` is complete in yacc (this warp's units and chunks):
    // add the sums of the row pair's other warps (one or three), then write Y or hand off.
    auto finish = [&](int tile, int seg_kb1) -> bool {
      const uint32_t ph_x = static_cast<uint32_t>(seg_count) & 1u;
      float* xb = xchg + (static_cast<size_t>(pr) * (2 * S::kPar - 1) * 32 + lane) * S::kXchgFloats;
      if (slot_id != 0) {
        // wait until the reader has taken the previous segment's values, then store ours
        if (seg_count > 0 && !mbar_wait(&xfree[pr], ph_x ^ 1u, wc)) return false;
        float* mine = xb + (slot_id - 1) * 32 * S::kXchgFloats;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int q = 0; q < NQ; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) mine[(j * NQ + q) * 4 + e] = yacc[j][q][e];
        __syncwarp();
        if (lane == 0) mbar_arrive(&xfull[pr]);
        return true;
      }
      if (!mbar_wait(&xfull[pr], ph_x, wc)) return false;
      float v[2][NQ][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int f = (j * NQ + q) * 4 + e;
            float a = yacc[j][q][e];
#pragma unroll
            for (int o = 0; o < 2 * S::kPar - 1; ++o) a += xb[o * 32 * S::kXchgFloats + f];
            v[j][q][e] = a;
          }
      __syncwarp();
      if (lane == 0) mbar_arrive(&xfree[pr]);
      // the tile's first weight row, first token row and token count (grouped: the expert's rows)
      int64_t n0 = static_cast<int64_t>(tile) * 128, y0 = 0;
      int tok_end = m_rows;
      if constexpr (MOE) {
        const TileInfo ti = decode_tile<MT, true>(p, tile, mtpre, moffs, kUnit);
        n0 = ti.n0;
        y0 = ti.m0;
        tok_end = ti.m_end - ti.m0;
      }
      auto store_y = [&](int j, int q, int e, float val) {
        const int tok = 8 * q + 2 * t + (e & 1);
        const int64_t row = n0 + rows[j][e >> 1];
        if (tok < tok_end && row < p.n) p.y[static_cast<size_t>(y0 + tok) * p.n + row] = __float2bfloat16_rn(val);
      };
      if (seg_kb0 == 0 && seg_kb1 == kb_total) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int q = 0; q < NQ; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) store_y(j, q, e, v[j][q][e]);
        return true;
      }
      if (csize > 1) {
        // Cluster hand-off: the cluster's CTAs are the tile's K ranges in order (rank 0 holds the
        // first k-block); ranks 1.. store their sums into rank 0's shared memory and arrive on its
        // barrier; rank 0 adds them in rank order (deterministic) and writes Y. One use per launch.
        constexpr int F = S::kXchgFloats;
        const uint32_t rank = blockIdx.x % static_cast<uint32_t>(csize);
        if (!cl_waited1) {
          cluster_wait();
          cl_waited1 = true;
        }
        if (rank != 0) {
          const uint32_t dst = map_to_rank(smem_u32(red + ((static_cast<size_t>(rank - 1) * 4 + pr) * 32 + lane) * F), 0);
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q)
              st_cluster_v4(dst + ((j * NQ + q) * 4) * 4, v[j][q][0], v[j][q][1], v[j][q][2], v[j][q][3]);
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(map_to_rank(smem_u32(&red_full[pr]), 0));
          cluster_arrive();
          cl_arrived2 = true;
          return true;
        }
        if (!mbar_wait_cluster(&red_full[pr], 0u, wc)) return false;
        cluster_arrive();
        cl_arrived2 = true;
        for (int r = 1; r < csize; ++r) {
          const float* src = red + ((static_cast<size_t>(r - 1) * 4 + pr) * 32 + lane) * F;
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q)
#pragma unroll
              for (int e = 0; e < 4; ++e) v[j][q][e] += src[(j * NQ + q) * 4 + e];
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int q = 0; q < NQ; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) store_y(j, q, e, v[j][q][e]);
        return true;
      }
      // Shared tile, fixed owner: the CTA holding the tile's first k-block (c_lo), which reaches
      // the tile at the end of its range, long after the others (c_lo+1 .. c_hi, for whom it is the
      // first segment) have published their fp32 partials [CTA][token][row].
      const int64_t it0 = static_cast<int64_t>(tile) * kb_total;
      const int64_t c_lo = sk_owner(it0, total, grid), c_hi = sk_owner(it0 + kb_total - 1, total, grid);
      uint32_t* ctr = sk_flag(p.counters, c_lo, pr);
      auto pidx = [&](int64_t c, int j, int q, int e) {
        const int tok = 8 * q + 2 * t + (e & 1);
        return static_cast<size_t>(c) * MT * 128 + static_cast<size_t>(tok) * 128 + rows[j][e >> 1];
      };
      if (static_cast<int64_t>(blockIdx.x) != c_lo) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int q = 0; q < NQ; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) __stcg(p.partial + pidx(blockIdx.x, j, q, e), v[j][q][e]);
        // the warp's stores are ordered before lane 0's release add (warp barrier, then release)
        __syncwarp();
        if (lane == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
        return true;
      }
      if (!sk_wait(ctr, static_cast<uint32_t>(c_hi - c_lo), wc)) return false;
      // own values first, then the other contributors in CTA order, CU of them in flight at a time
      constexpr int CU = NQ == 1 ? 4 : 2;
      for (int64_t c = c_lo + 1; c <= c_hi; c += CU) {
        float pv[CU][2][NQ][4];
#pragma unroll
        for (int uu = 0; uu < CU; ++uu) {
          const int64_t cc = c + uu <= c_hi ? c + uu : c_hi;
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q)
#pragma unroll
              for (int e = 0; e < 4; ++e) pv[uu][j][q][e] = __ldcg(p.partial + pidx(cc, j, q, e));
        }
#pragma unroll
        for (int uu = 0; uu < CU; ++uu) {
          if (c + uu > c_hi) break;
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int q = 0; q < NQ; ++q)
#pragma unroll
              for (int e = 0; e < 4; ++e) v[j][q][e] += pv[uu][j][q][e];
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) store_y(j, q, e, v[j][q][e]);
      __syncwarp();
      if (lane == 0) *ctr = 0u;   // for the next call (no contributor touches it again in this one)
      return true;
    };

    // Segments (the parts of tiles in this CTA's range) in order; within each, this warp's units.
    int i = par, s = par;                      // unit ordinal in the range, its stage
    uint32_t ph = 0;
    int tile = tile0;
    for (int seg_end = 0; seg_end < n_units; ++tile) {
      const int seg_begin = seg_end;
      seg_end = seg_begin + (kb_total - seg_kb0 < n_units - seg_begin ? kb_total - seg_kb0 : n_units - seg_begin);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) yacc[j][q][e] = 0.f;
      bool ok = true;
      for (; i < seg_end; i += S::kPar) {
        if (!mbar_wait(&full[s], ph, wc) || ((WK == 0 || WK == 8) && !mbar_wait(&meta_full[s], ph, wc))) { ok = false; break; }
        if (cw == 0 && lane == 0 && i == 0) trace_mark(p.trace, 4);
        const uint32_t base = smem0 + s * S::kStage;
        uint32_t bx[NQ][2][4];
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint4 v = ld_shared_v4(base + xoff + q * 8 * S::kXPitch + cc * 64);
            bx[q][cc][0] = v.x; bx[q][cc][1] = v.y; bx[q][cc][2] = v.z; bx[q][cc][3] = v.w;
          }
        uint32_t wd[2][2][2];
        if constexpr (WK != 8) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) wd[j][hl][cc] = lds32(base + woff + cc * 2048 + j * 256 + hl * 128);
        }
        if constexpr (WK == 8) {
          // the lane's 8 codes of each row and 32-K chunk: bytes 8 (t % 2) .. of 16-column slot
          // 2 (chunk) + t / 2; exact integers u - z, the block's scale applied to the sums
          float sc[2][2], zf[2][2];
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) {
              uint32_t sb, zb;
              asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(sb), "=r"(zb) : "r"(base + moff + j * 128 + hl * 64));
              sc[j][hl] = __uint_as_float(sb);
              zf[j][hl] = __uint_as_float(zb);
            }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float d[2][NQ][4];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              uint32_t lo[4], hi[4];
#pragma unroll
              for (int hl = 0; hl < 2; ++hl) {
                const uint32_t rr = static_cast<uint32_t>(32 * pr + g + 16 * j + 8 * hl);
                uint32_t w0, w1;
                asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                             : "=r"(w0), "=r"(w1)
                             : "r"(base + (2 * (2 * cp + cc) + (t >> 1)) * 2048 + rr * 16 + 8 * (t & 1)));
                uint32_t e0[2], e1[2];
                dq_int8_word_unscaled(w0, zf[j][hl], e0);
                dq_int8_word_unscaled(w1, zf[j][hl], e1);
                uint32_t* dst = hl ? hi : lo;
                dst[0] = e0[0]; dst[1] = e0[1]; dst[2] = e1[0]; dst[3] = e1[1];
              }
#pragma unroll
              for (int q = 0; q < NQ; ++q) {
                mma_bf16_16816_z(d[cc][q], lo[0], hi[0], lo[1], hi[1], bx[q][cc][0], bx[q][cc][1]);
                mma_bf16_16816(d[cc][q], lo[2], hi[2], lo[3], hi[3], bx[q][cc][2], bx[q][cc][3]);
              }
            }
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
              yacc[j][q][0] = fmaf(sc[j][0], d[0][q][0] + d[1][q][0], yacc[j][q][0]);
              yacc[j][q][1] = fmaf(sc[j][0], d[0][q][1] + d[1][q][1], yacc[j][q][1]);
              yacc[j][q][2] = fmaf(sc[j][1], d[0][q][2] + d[1][q][2], yacc[j][q][2]);
              yacc[j][q][3] = fmaf(sc[j][1], d[0][q][3] + d[1][q][3], yacc[j][q][3]);
            }
          }
        } else if constexpr (G32) {
          // per (row, 32-K chunk): bf16 scales of chunks 2cp, 2cp + 1 in one word, u4 zero-points
          // of the row's four chunks in one half-word
          uint32_t sw[2][2], zw[2][2];
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) {
              const uint32_t rr = static_cast<uint32_t>(32 * pr + g + 16 * j + 8 * hl);
              sw[j][hl] = lds32(base + kUnitCodes + rr * 8 + 4 * cp);
              uint32_t zb = 0x8888u;
              if (has_zero) {
                uint16_t h16;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h16) : "r"(base + kUnitG32 + rr * 2));
                zb = h16;
              }
              zw[j][hl] = zb >> (8 * cp);   // chunks 2cp, 2cp + 1 in the low byte
            }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float d[2][NQ][4];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              uint32_t lo[4], hi[4];
              const uint32_t zl = (zw[j][0] >> (4 * cc)) & 0xFu, zh = (zw[j][1] >> (4 * cc)) & 0xFu;
              dq_int4_word_unscaled(wd[j][0][cc], 0x43004300u | zl | (zl << 16), lo);
              dq_int4_word_unscaled(wd[j][1][cc], 0x43004300u | zh | (zh << 16), hi);
#pragma unroll
              for (int q = 0; q < NQ; ++q) {
                mma_bf16_16816_z(d[cc][q], lo[0], hi[0], lo[1], hi[1], bx[q][cc][0], bx[q][cc][1]);
                mma_bf16_16816(d[cc][q], lo[2], hi[2], lo[3], hi[3], bx[q][cc][2], bx[q][cc][3]);
              }
            }
            const float s00 = __uint_as_float(sw[j][0] << 16), s01 = __uint_as_float(sw[j][0] & 0xFFFF0000u);
            const float s10 = __uint_as_float(sw[j][1] << 16), s11 = __uint_as_float(sw[j][1] & 0xFFFF0000u);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
              yacc[j][q][0] = fmaf(s01, d[1][q][0], fmaf(s00, d[0][q][0], yacc[j][q][0]));
              yacc[j][q][1] = fmaf(s01, d[1][q][1], fmaf(s00, d[0][q][1], yacc[j][q][1]));
              yacc[j][q][2] = fmaf(s11, d[1][q][2], fmaf(s10, d[0][q][2], yacc[j][q][2]));
              yacc[j][q][3] = fmaf(s11, d[1][q][3], fmaf(s10, d[0][q][3], yacc[j][q][3]));
            }
          }
        } else if constexpr (!MX) {
          float sc[2][2];
          uint32_t z2[2][2];
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) {
              uint32_t sb, zb;
              asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(sb), "=r"(zb) : "r"(base + moff + j * 128 + hl * 64));
              sc[j][hl] = __uint_as_float(sb);
              z2[j][hl] = zb;
            }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float d[2][NQ][4];   // per chunk: two short MMA chains instead of one long one
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              uint32_t lo[4], hi[4];
              dq_int4_word_unscaled(wd[j][0][cc], z2[j][0], lo);
              dq_int4_word_unscaled(wd[j][1][cc], z2[j][1], hi);
#pragma unroll
              for (int q = 0; q < NQ; ++q) {
                mma_bf16_16816_z(d[cc][q], lo[0], hi[0], lo[1], hi[1], bx[q][cc][0], bx[q][cc][1]);
                mma_bf16_16816(d[cc][q], lo[2], hi[2], lo[3], hi[3], bx[q][cc][2], bx[q][cc][3]);
              }
            }
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
              yacc[j][q][0] = fmaf(sc[j][0], d[0][q][0] + d[1][q][0], yacc[j][q][0]);
              yacc[j][q][1] = fmaf(sc[j][0], d[0][q][1] + d[1][q][1], yacc[j][q][1]);
              yacc[j][q][2] = fmaf(sc[j][1], d[0][q][2] + d[1][q][2], yacc[j][q][2]);
              yacc[j][q][3] = fmaf(sc[j][1], d[0][q][3] + d[1][q][3], yacc[j][q][3]);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint32_t e4[2];
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) e4[hl] = lds32(base + moff + j * 64 + hl * 32);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              uint32_t a[2][4];
#pragma unroll
              for (int hl = 0; hl < 2; ++hl) {
                const uint32_t ex = (e4[hl] >> (8 * (2 * cp + cc))) & 0xFFu;
                if constexpr (WK == 3) {
                  dq_int4_word(wd[j][hl][cc], int4_zero_pair(8), bits_bf16x2(mxint_scale_pair(ex)), a[hl]);
                } else if (ex <= 128u) {
                  dq_mx_word_bits(wd[j][hl][cc], mx_pow2_pair(ex), a[hl]);
                } else {
                  dq_mx_word(wd[j][hl][cc], lut, pow2f(static_cast<int>(ex) - 127), a[hl]);
                }
              }
#pragma unroll
              for (int q = 0; q < NQ; ++q) {
                mma_bf16_16816(yacc[j][q], a[0][0], a[1][0], a[0][1], a[1][1], bx[q][cc][0], bx[q][cc][1]);
                mma_bf16_16816(yacc[j][q], a[0][2], a[1][2], a[0][3], a[1][3], bx[q][cc][2], bx[q][cc][3]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        s += S::kPar;
        if (s >= SL) { s -= SL; ph ^= 1u; }
      }
      if (!ok) break;
      if (cw == 0 && lane == 0 && seg_end == n_units) trace_mark(p.trace, 7);
      // every warp closes every segment, even one without a unit of its parity
      if (!finish(tile, seg_kb0 + (seg_end - seg_begin))) break;
      if (cw == 0 && lane == 0 && seg_end == n_units) trace_mark(p.trace, 9);
      ++seg_count;
      seg_kb0 = 0;
    }
  }
  if (lane == 0) trace_stage(p.trace, 0, warp);   // (diagnostics: when each warp finished its role)
  // no CTA leaves while another of its cluster may still write into its shared memory
  if (csize > 1) {
    if (!cl_waited1) cluster_wait();
    if (!cl_arrived2) cluster_arrive();
    cluster_wait();
  }
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0) trace_mark(p.trace, 12);
}

template <int MT, int WK>
cudaError_t launch_v(const F16Params& p_in, cudaStream_t st) {
  using S = VShape<MT, v_wbytes(WK)>;
  auto kern = gemv_kernel<MT, WK, false>;
  static int configured[64] = {};
  static int cluster_max[64][kVMaxCluster + 1] = {};   // active clusters the device holds, +1 (0 unknown)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  F16Params p = p_in;
  // Cluster hand-off when every tile is cut into 2..4 K ranges, one per CTA (grid = tiles x ranges),
  // and the device can hold all the clusters at once (they wait on each other).
  const int32_t tiles = p.sched.num_tiles, grid = p.sched.grid;
  const int ranges = tiles > 0 && grid % tiles == 0 ? grid / tiles : 0;
  int cs = ranges >= 2 && ranges <= kVMaxCluster && ranges <= p.sched.kb_total ? ranges : 1;
  static const bool clusters_on = [] {   // HM_GEMV_CLUSTER=0: the global-memory hand-off everywhere
    const char* v = std::getenv("HM_GEMV_CLUSTER");
    return !(v && v[0] == '0');
  }();
  if (!clusters_on) cs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(v_threads(MT)));
  cfg.dynamicSmemBytes = static_cast<size_t>(S::kSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  if (cs > 1 && cluster_max[dev][cs] == 0) {
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    cluster_max[dev][cs] = n + 1;
  }
  if (cs > 1 && (cluster_max[dev][cs] - 1) * cs < grid) cs = 1;   // not all clusters fit at once
  p.cluster = cs;
  if (cs <= 1) return launch_pdl(kern, grid, v_threads(MT), S::kSmem, st, p);
  static const bool pdl = [] {
    const char* v = std::getenv("HM_PDL");
    return !(v && v[0] == '0');
  }();
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Grouped variant: persistent CTAs over the stream-K range of all experts' (token tile, weight
// tile, k-block) units; no clusters (the tile count is known only on the device).
template <int MT, int WK>
cudaError_t launch_vm(const F16Params& p, cudaStream_t st) {
  using S = VShape<MT, v_wbytes(WK), true>;
  auto kern = gemv_kernel<MT, WK, true>;
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return launch_pdl(kern, p.sched.grid, v_threads(MT), S::kSmem, st, p);
}

}  // namespace

int gemv_tokens(int64_t m) { return m <= 8 ? 8 : (m <= 16 ? 16 : 32); }

int gemv_stages(int64_t m, int32_t fmt) {
  const int t = gemv_tokens(m);
  if (fmt == kW4A16Int4G)
    return t == 8 ? VShape<8, v_wbytes(6)>::kS : (t == 16 ? VShape<16, v_wbytes(6)>::kS : VShape<32, v_wbytes(6)>::kS);
  if (fmt == kW8A16Int8)
    return t == 8 ? VShape<8, v_wbytes(8)>::kS : (t == 16 ? VShape<16, v_wbytes(8)>::kS : VShape<32, v_wbytes(8)>::kS);
  return t == 8 ? VShape<8>::kS : (t == 16 ? VShape<16>::kS : VShape<32>::kS);
}

cudaError_t launch_gemv(const F16Params& p, cudaStream_t st) {
  if (p.m < 1 || p.m > kGemvMaxTokens) return cudaErrorInvalidValue;
  const int t = gemv_tokens(p.m);
  if (p.fmt == kW4A16Mx)
    return t == 8 ? launch_v<8, 2>(p, st) : (t == 16 ? launch_v<16, 2>(p, st) : launch_v<32, 2>(p, st));
  if (p.fmt == kW4A16MxInt)
    return t == 8 ? launch_v<8, 3>(p, st) : (t == 16 ? launch_v<16, 3>(p, st) : launch_v<32, 3>(p, st));
  if (p.fmt == kW4A16Int4G)
    return t == 8 ? launch_v<8, 6>(p, st) : (t == 16 ? launch_v<16, 6>(p, st) : launch_v<32, 6>(p, st));
  if (p.fmt == kW8A16Int8)
    return t == 8 ? launch_v<8, 8>(p, st) : (t == 16 ? launch_v<16, 8>(p, st) : launch_v<32, 8>(p, st));
  return t == 8 ? launch_v<8, 0>(p, st) : (t == 16 ? launch_v<16, 0>(p, st) : launch_v<32, 0>(p, st));
}

cudaError_t launch_gemv_moe(const F16Params& p, int tokens, cudaStream_t st) {
  if (p.num_experts < 1 || p.num_experts > kGemvMoeMaxExperts || p.k % 128 != 0 || (tokens != 8 && tokens != 16))
    return cudaErrorInvalidValue;
  const bool t8 = tokens == 8;
  switch (p.fmt) {
    case kW4A16Int4: return t8 ? launch_vm<8, 0>(p, st) : launch_vm<16, 0>(p, st);
    case kW4A16Mx: return t8 ? launch_vm<8, 2>(p, st) : launch_vm<16, 2>(p, st);
    case kW4A16MxInt: return t8 ? launch_vm<8, 3>(p, st) : launch_vm<16, 3>(p, st);
    case kW4A16Int4G: return t8 ? launch_vm<8, 6>(p, st) : launch_vm<16, 6>(p, st);
    case kW8A16Int8: return t8 ? launch_vm<8, 8>(p, st) : launch_vm<16, 8>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hm
