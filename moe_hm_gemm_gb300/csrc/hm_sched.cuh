// Work schedules shared by the persistent GEMM kernels.
//
// A tile is 128 weight rows x `tile_m` tokens; its K loop has `kb_total` k-blocks. Modes:
//  * tile-parallel: CTA b takes tiles b, b+G, b+2G, ... with their whole K loop;
//  * stream-K (small M, fewer tiles than SMs): the flattened (tile, k-block) space of
//    num_tiles*kb_total iterations is cut into G contiguous ranges, start(c) =
//    floor(c*total/G); a CTA's range crosses tile boundaries, so a tile may be shared by
//    several CTAs, each producing an fp32 partial that the tile's owner (the CTA holding its
//    first k-block) sums in k order (fixed-owner hand-off below). G <= total guarantees every
//    range is non-empty, so the number of CTAs sharing a tile is exactly c_hi - c_lo + 1;
//  * hybrid (sk_tiles = S, 0 < S < num_tiles, with stream-K): the first S tiles (the remainder
//    of num_tiles over G, which tile-parallel waves would leave to a partly filled last wave) are
//    cut into stream-K ranges as above over S*kb_total iterations (G <= S*kb_total), and every
//    CTA then takes tiles S + b, S + b + G, ... whole. The stream-K part comes first, so its
//    shared tiles are handed off as in plain stream-K; the tiles it covers are the first token
//    tiles, few enough for their activations to stay in L2 while they are split.
#pragma once
#include <cstdint>

#include "hm_device.cuh"

namespace hm {

struct SchedParams {
  int32_t num_tiles;
  int32_t kb_total;
  int32_t grid;
  int32_t stream_k;
  int32_t sk_tiles;   // with stream_k: tiles cut into stream-K ranges before the tile-parallel rest
                      // (0 or >= num_tiles: all of them)
};

// Tiles the stream-K ranges cover (the hand-off below indexes the flattened space of these).
__host__ __device__ __forceinline__ int32_t sk_tiles_of(const SchedParams& s, int32_t num_tiles) {
  if (s.stream_k == 0) return 0;
  return (s.sk_tiles > 0 && s.sk_tiles < num_tiles) ? s.sk_tiles : num_tiles;
}

__host__ __device__ __forceinline__ int64_t sk_start(int64_t c, int64_t total, int64_t g) {
  return c * total / g;
}

// CTA whose stream-K range contains iteration `it`.
__host__ __device__ __forceinline__ int64_t sk_owner(int64_t it, int64_t total, int64_t g) {
  int64_t c = it * g / total;
  while (c + 1 < g && sk_start(c + 1, total, g) <= it) ++c;
  while (c > 0 && sk_start(c, total, g) > it) --c;
  return c;
}

// Arrival counters of a shared tile belong to its owner CTA: a CTA owns at most one shared tile
// (the last segment of its contiguous range), so [grid][kCounterSlots] counters serve every problem
// size, and a workspace's counters never move with the problem (calls of any size and entry may
// share one workspace: no call's partials or activations land on another call's counters).
constexpr int kCounterSlots = 8;

__device__ __forceinline__ uint32_t* sk_flag(uint32_t* counters, int64_t owner_cta, int slot) {
  return counters + static_cast<size_t>(owner_cta) * kCounterSlots + slot;
}

// Owner CTA of `tile` (the one whose range holds its first k-block).
__host__ __device__ __forceinline__ int64_t sk_tile_owner(int32_t tile, int32_t kb_total, int64_t total, int64_t g) {
  return sk_owner(static_cast<int64_t>(tile) * kb_total, total, g);
}

struct Segment {
  int32_t tile;
  int32_t kb0;
  int32_t kb1;
};

// Cursor over a CTA's segments. The (tile, k-block) space has fewer than 2^31 iterations (the
// API bounds M, N and K), so the per-segment steps divide in 32 bits; only the range ends, whose
// products c * total can exceed 2^31, are computed in 64 bits, once. (A 64-bit division is a
// long instruction sequence, and every role walks the schedule at start-up.)
struct SchedIter {
  int32_t it, it_end;     // stream-K cursor
  int32_t next_tile;      // tile-parallel cursor (after the stream-K tiles)
  int32_t stride;
  int32_t num_tiles;
  int32_t kb_total;

  __device__ __forceinline__ void init(const SchedParams& s, int32_t num_tiles_override, int32_t b) {
    num_tiles = num_tiles_override;
    kb_total = s.kb_total;
    stride = s.grid;
    const int32_t sk_n = sk_tiles_of(s, num_tiles);
    next_tile = sk_n + b;
    if (sk_n > 0) {
      const int64_t total = static_cast<int64_t>(sk_n) * kb_total;
      it = static_cast<int32_t>(sk_start(b, total, s.grid));
      it_end = static_cast<int32_t>(sk_start(b + 1, total, s.grid));
    } else {
      it = it_end = 0;
    }
  }

  __device__ __forceinline__ bool next(Segment& seg) {
    if (it < it_end) {
      const uint32_t q = static_cast<uint32_t>(it) / static_cast<uint32_t>(kb_total);
      seg.tile = static_cast<int32_t>(q);
      seg.kb0 = it - static_cast<int32_t>(q) * kb_total;
      const int32_t left = it_end - it;
      seg.kb1 = seg.kb0 + left < kb_total ? seg.kb0 + left : kb_total;
      it += seg.kb1 - seg.kb0;
      return true;
    }
    if (next_tile >= num_tiles) return false;
    seg.tile = next_tile;
    seg.kb0 = 0;
    seg.kb1 = kb_total;
    next_tile += stride;
    return true;
  }
};

// ---------------------------------------------------------------------------------------
// Fixed-owner hand-off of a stream-K tile. The owner is the CTA whose range holds the tile's
// first k-block (segment with kb0 == 0). In forward stream-K order that is the last segment of
// its range, while every other contributor holds the tile in the first segment of its own range,
// so by the time the owner finishes, the others have long published. Non-owners store their
// fp32 partial rows ([cta][first/last segment][row][tile_m]) and add 1 to the owner's per-warp
// flag (sk_flag) with release semantics, without waiting for anything; the owner waits (bounded) until the
// flag shows all of them, adds their partials to its own in k order (CTA c_lo = itself first,
// so the sum is deterministic), writes Y and clears the flag for the next call.

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Non-owner: publish this warp's partial rows (already stored by every lane).
__device__ __forceinline__ void sk_publish(uint32_t* flag, int lane) {
  __threadfence();
  __syncwarp();
  if (lane == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(flag) : "memory");
}

// Owner: wait until `expect` contributors have published. Every lane polls with an acquire load,
// so its later loads of the partials are ordered after the flag. False when the CTA is aborting
// or the wait ran out (then kErrTimeout and the abort flag are set).
__device__ __forceinline__ bool sk_wait(const uint32_t* flag, uint32_t expect, const WaitCtx& ctx) {
  if (ld_acquire_gpu(flag) >= expect) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (ld_acquire_gpu(flag) >= expect) return true;
    if (*ctx.abort) return false;
    if (globaltimer() - t0 > ctx.timeout_ns) {
      *ctx.abort = 1u;
      atomicOr(ctx.err, kErrTimeout);
      return false;
    }
  }
}

// Row `row` of the partial that CTA c stored for `tile` ([cta][first/last segment][row][BT]): its
// first slot when its range starts in that tile.
template <int BT>
__device__ __forceinline__ const float* sk_partial_row(const float* partial, int64_t total_it, int32_t grid,
                                                       int32_t kb_total, int32_t tile, int64_t c, int row) {
  const int which = (sk_start(c, total_it, grid) / kb_total == tile) ? 0 : 1;
  return partial + (static_cast<size_t>(c) * 2 + which) * BT * 128 + static_cast<size_t>(row) * BT;
}

// Owner: add columns [j0, j0 + 16) of the other contributors' partial rows (CTAs c_lo+1 .. c_hi,
// in that order) to `acc`, which holds the owner's own values. Loads of up to four contributors
// are in flight together.
template <int BT>
__device__ __forceinline__ void sk_add_partials(const float* partial, int64_t total_it, int32_t grid,
                                                int32_t kb_total, int32_t tile, int64_t c_lo, int64_t c_hi,
                                                int row, int j0, float (&acc)[16]) {
  auto src = [&](int64_t c) {
    return reinterpret_cast<const float4*>(sk_partial_row<BT>(partial, total_it, grid, kb_total, tile, c, row) + j0);
  };
  int64_t c = c_lo + 1;
#pragma unroll 1
  for (; c + 3 <= c_hi; c += 4) {
    float4 v[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4* s4 = src(c + u);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[u][i] = __ldcg(s4 + i);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[4 * i] += v[u][i].x;
        acc[4 * i + 1] += v[u][i].y;
        acc[4 * i + 2] += v[u][i].z;
        acc[4 * i + 3] += v[u][i].w;
      }
    }
  }
#pragma unroll 1
  for (; c <= c_hi; ++c) {
    const float4* s4 = src(c);
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldcg(s4 + i);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[4 * i] += v[i].x;
      acc[4 * i + 1] += v[i].y;
      acc[4 * i + 2] += v[i].z;
      acc[4 * i + 3] += v[i].w;
    }
  }
}

}  // namespace hm
