// Work schedules shared by the persistent GEMM kernels.
//
// A tile is 128 weight rows x `tile_m` tokens; its K loop has `kb_total` k-blocks. Two modes:
//  * tile-parallel: CTA b takes tiles b, b+G, b+2G, ... with their whole K loop;
//  * stream-K (small M, fewer tiles than SMs): the flattened (tile, k-block) space of
//    num_tiles*kb_total iterations is cut into G contiguous ranges, start(c) =
//    floor(c*total/G); a CTA's range crosses tile boundaries, so a tile may be shared by
//    several CTAs, each producing an fp32 partial that one of them (the last to finish,
//    found with an atomic counter) sums in k order. G <= total guarantees every range is
//    non-empty, so the number of CTAs sharing a tile is exactly c_hi - c_lo + 1.
#pragma once
#include <cstdint>

namespace hm {

struct SchedParams {
  int32_t num_tiles;
  int32_t kb_total;
  int32_t grid;
  int32_t stream_k;
};

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

struct Segment {
  int32_t tile;
  int32_t kb0;
  int32_t kb1;
};

struct SchedIter {
  int64_t it, it_end;     // stream-K cursor
  int32_t next_tile;      // tile-parallel cursor
  int32_t stride;
  int32_t num_tiles;
  int32_t kb_total;
  bool stream_k;

  __device__ __forceinline__ void init(const SchedParams& s, int32_t num_tiles_override, int32_t b) {
    num_tiles = num_tiles_override;
    kb_total = s.kb_total;
    stream_k = s.stream_k != 0;
    stride = s.grid;
    next_tile = b;
    const int64_t total = static_cast<int64_t>(num_tiles) * kb_total;
    it = sk_start(b, total, s.grid);
    it_end = sk_start(b + 1, total, s.grid);
  }

  __device__ __forceinline__ bool next(Segment& seg) {
    if (stream_k) {
      if (it >= it_end) return false;
      seg.tile = static_cast<int32_t>(it / kb_total);
      seg.kb0 = static_cast<int32_t>(it % kb_total);
      const int64_t left = it_end - it;
      seg.kb1 = static_cast<int32_t>(seg.kb0 + left < kb_total ? seg.kb0 + left : kb_total);
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

// Sum the stream-K partials of one tile for one accumulator row, in k order (CTA c_lo first),
// and hand each column's total to `emit(j, value)`. Partials are laid out
// [cta][first/last segment][row][tile_m] (fp32), so each lane reads its row's columns with
// 16-byte loads; four contributors' loads are issued before any of them is summed, which keeps
// many independent L2 reads in flight instead of one dependent read per column.
template <int BT, typename Emit>
__device__ __forceinline__ void streamk_fixup(const float* partial, int64_t total_it, int32_t grid,
                                              int32_t kb_total, int32_t tile, int64_t c_lo, int64_t c_hi,
                                              int row, Emit emit) {
  auto src = [&](int64_t c) {
    const int which = (sk_start(c, total_it, grid) / kb_total == tile) ? 0 : 1;
    return partial + (static_cast<size_t>(c) * 2 + which) * BT * 128 + static_cast<size_t>(row) * BT;
  };
#pragma unroll 1
  for (int j0 = 0; j0 < BT; j0 += 16) {
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    int64_t c = c_lo;
#pragma unroll 1
    for (; c + 3 <= c_hi; c += 4) {
      float4 v[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4* s4 = reinterpret_cast<const float4*>(src(c + u) + j0);
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
      const float4* s4 = reinterpret_cast<const float4*>(src(c) + j0);
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
#pragma unroll
    for (int i = 0; i < 16; ++i) emit(j0 + i, acc[i]);
  }
}

}  // namespace hm
