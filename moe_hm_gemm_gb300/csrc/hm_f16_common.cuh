// Pieces shared by the two W4A16 GEMM kernels (the general one in hm_gemm_f16.cu and the
// small-token INT4 one in hm_gemm_f16s.cu): tile decoding for the dense and the grouped MoE
// schedules, header validation, the MoE tile prefix, bounded draining, and the store of a
// finished tile (direct, or as a stream-K partial with its fix-up).
#pragma once
#include <cuda_bf16.h>

#include "hm_device.cuh"
#include "hm_kernels.h"
#include "hm_layout.h"
#include "hm_sched.cuh"

namespace hm {
namespace {

struct TileInfo {
  int32_t m0, m_end, n0;
  const uint8_t* base;   // packed weight (header) of this tile's matrix
  const uint8_t* wbase;  // first unit of this n-tile
};

// Largest e with prefix[e] <= tile (prefix[0] = 0 <= tile < prefix[E]).
__device__ __forceinline__ int find_expert(const int32_t* prefix, int experts, int tile) {
  int lo = 0, hi = experts;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  return lo;
}

template <int BT, bool MOE>
__device__ __forceinline__ TileInfo decode_tile(const F16Params& p, int tile, const int32_t* prefix,
                                                const int32_t* offs, uint32_t unit) {
  TileInfo t;
  const int64_t kb_total = p.k / 128;
  if (!MOE) {
    // m-major: concurrent CTAs share one X tile and stream different weight tiles; or grouped
    // (group_m > 1): within a group of group_m token tiles the token tile changes fastest, so a wave
    // covers group_m token tiles and about CTAs / group_m weight tiles
    int nt, mt;
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
    t.m0 = mt * BT;
    t.m_end = static_cast<int32_t>(p.m < t.m0 + BT ? p.m : t.m0 + BT);
    t.n0 = nt * 128;
    t.base = p.packed;
    t.wbase = p.packed + kHeaderBytes + static_cast<size_t>(nt) * kb_total * unit;
  } else {
    const int e = find_expert(prefix, p.num_experts, tile);
    const int local = tile - prefix[e];
    // m-major within the expert, as in the dense order: the CTAs of one wave share an X tile and
    // stream the expert's weight tiles, which stay in L2 while its token tiles are processed (the
    // other order re-reads a heavy expert's X rows, hundreds of MB, once per weight tile)
    const int nt = local % p.num_n_tiles;
    const int mt = local / p.num_n_tiles;
    t.m0 = offs[e] + mt * BT;
    t.m_end = min(offs[e + 1], t.m0 + BT);
    t.n0 = nt * 128;
    t.base = p.packed_list != nullptr ? p.packed_list[e] : p.packed + static_cast<size_t>(e) * p.expert_stride;
    t.wbase = t.base + kHeaderBytes + static_cast<size_t>(nt) * kb_total * unit;
  }
  return t;
}

__device__ __forceinline__ bool header_ok(const uint8_t* packed, const F16Params& p, uint32_t has_zero) {
  const PackedHeader* h = reinterpret_cast<const PackedHeader*>(packed);
  return h->magic == kMagic && static_cast<int32_t>(h->fmt) == p.fmt && h->n == p.n &&
         h->k == p.k && h->has_zero == has_zero;
}

// Wait without looking at the abort flag (used to drain in-flight work before exit).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}


// MoE: per-expert tile counts and their exclusive prefix over the expert-sorted offsets, computed
// by one warp; offsets are copied to shared memory. Malformed offsets (decreasing, negative,
// beyond M, or not starting at 0) set kErrOffsets and the abort flag.
template <int BT>
__device__ __forceinline__ void moe_tile_prefix(const F16Params& p, int32_t* offs, int32_t* prefix,
                                                volatile uint32_t* abort_flag, int lane) {
  const int E = p.num_experts;
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
  if (__any_sync(0xffffffffu, bad) && lane == 0) {
    atomicOr(p.err, kErrOffsets);
    *abort_flag = 1u;
  }
}

// Store one weight row's finished segment of a tile: `acc[j]` is the fp32 sum over the segment's
// k-blocks for token m0 + j. A segment covering the whole K loop writes Y (bf16, rounded once).
// Otherwise the tile is shared by stream-K CTAs c_lo .. c_hi: a non-owner stores its partial rows
// and publishes them; the owner (the segment holding k-block 0) waits for the others, adds their
// partials to its own in k order and writes Y (see the fixed-owner hand-off in hm_sched.cuh).
template <int BT>
__device__ __forceinline__ void store_segment(const F16Params& p, const TileInfo& t, const Segment& seg,
                                              int kb_total, int64_t total_it, bool first_seg, int q, int lane,
                                              const WaitCtx& wc, const float (&acc)[BT]) {
  const int row = 32 * q + lane;
  const int64_t n = static_cast<int64_t>(t.n0) + row;
  auto emit = [&](int j, float v) {
    const int64_t m = static_cast<int64_t>(t.m0) + j;
    if (m < t.m_end && n < p.n) p.y[m * p.n + n] = __float2bfloat16_rn(v);
  };
  if (seg.kb0 == 0 && seg.kb1 == kb_total) {
#pragma unroll
    for (int j = 0; j < BT; ++j) emit(j, acc[j]);
    return;
  }
  uint32_t* flag = sk_flag(p.counters, seg.kb0 == 0 ? blockIdx.x : sk_tile_owner(seg.tile, kb_total, total_it,
                                                                                 p.sched.grid), q);
  if (seg.kb0 != 0) {
    float* slot = p.partial + (static_cast<size_t>(blockIdx.x) * 2 + (first_seg ? 0 : 1)) * BT * 128 +
                  static_cast<size_t>(row) * BT;
#pragma unroll
    for (int j = 0; j < BT; j += 4)
      *reinterpret_cast<float4*>(slot + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
    sk_publish(flag, lane);
    if (row == 0) trace_mark(p.trace, 10);
    return;
  }
  const int64_t c_lo = blockIdx.x;
  const int64_t c_hi = sk_owner(static_cast<int64_t>(seg.tile + 1) * kb_total - 1, total_it, p.sched.grid);
  if (!sk_wait(flag, static_cast<uint32_t>(c_hi - c_lo), wc)) return;
  if (row == 0) trace_mark(p.trace, 10);
#pragma unroll
  for (int j0 = 0; j0 < BT; j0 += 16) {
    float a[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) a[j] = acc[j0 + j];
    sk_add_partials<BT>(p.partial, total_it, p.sched.grid, kb_total, seg.tile, c_lo, c_hi, row, j0, a);
#pragma unroll
    for (int j = 0; j < 16; ++j) emit(j0 + j, a[j]);
  }
  __syncwarp();
  if (lane == 0) *flag = 0u;
  if (row == 0) trace_mark(p.trace, 11);
}

}  // namespace
}  // namespace hm
