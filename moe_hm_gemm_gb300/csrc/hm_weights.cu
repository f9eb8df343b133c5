// Weight-side kernels: round-to-nearest quantization of fp32 weights into the standard
// format, the one-time transform (pad + relayout) into the packed layout the GEMM kernels
// stream, and the dequant test hook.
//
// Method references: the explainer page "vLLM Humming은 4비트를 어떻게 계산하나", section
// "4비트 값에는 스케일이라는 해석 규칙이 붙는다" (q = round(w/s) in [-8, 7], restored s*q, one
// 16-bit scale per 128 weights) and section "표현을 맞춘 다음 GPU가 읽기 좋은 배치로 바꾼다"
// (weights, scales and zero-points are padded and rearranged once for the device). MXFP4
// follows OCP Microscaling v1.0; MXINT4 takes the same shared exponent with signed 4-bit integer
// elements; NVFP4 the two-level (e4m3 per 16, fp32 per tensor) recipe.
#include <cuda_bf16.h>

#include "hm_dequant.cuh"
#include "hm_device.cuh"
#include "hm_kernels.h"
#include "hm_layout.h"

namespace hm {
namespace {

__device__ __forceinline__ float warp_max(float v, int width) {
  for (int d = width / 2; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

// fp32 pair -> e2m1 pair in one byte (RNE, saturating); `lo` goes to the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u16.u8 %0, b;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// fp32 -> e4m3 code (RNE, saturating).
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
  return r & 0xFFu;
}

// e4m3 code -> value (exact), from the bit fields (bias 7, 3 mantissa bits, subnormals).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float mag = e == 0 ? static_cast<float>(m) * 0.001953125f  // m * 2^-9
                           : static_cast<float>(8u + m) * pow2f(static_cast<int>(e) - 10);
  return (c & 0x80u) ? -mag : mag;
}

// ------------------------------------------------------------------ quantization (standard format)

// INT4 with a bf16 scale per group of `group` along K (32, 64, or a multiple of 128): one warp per
// (row, group of max(group, 128) K); lane holds 4 consecutive K of each 128-K chunk. A group of 32
// or 64 is the amax over its 8 or 16 lanes; a group of 128 j takes the amax over its j chunks
// first, then quantizes them.
__global__ void quant_int4_kernel(const float* __restrict__ w, const uint8_t* __restrict__ zeros,
                                  int64_t n, int64_t k, int has_zero, int64_t group, uint8_t* __restrict__ q,
                                  __nv_bfloat16* __restrict__ scales) {
  const int64_t span = group < 128 ? 128 : group;        // K per warp
  const int64_t spans = k / span;
  const int64_t gid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gid >= n * spans) return;
  const int64_t row = gid / spans, sp = gid % spans;
  const int64_t groups = k / group;
  const int width = group < 128 ? static_cast<int>(group / 4) : 32;   // lanes per group within a chunk
  float amax = 0.f;
  for (int64_t c = 0; c < span / 128; ++c) {
    const float4 v = *reinterpret_cast<const float4*>(w + row * k + sp * span + c * 128 + 4 * lane);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  amax = warp_max(amax, width);
  const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(amax, 7.0f));
  const float s = __bfloat162float(sb);
  // the group of this lane's values (the same for every chunk of a wide group)
  const int64_t gi = group < 128 ? (sp * 128 + 4 * lane) / group : sp;
  const int z = has_zero ? zeros[row * groups + gi] : 0;
  for (int64_t c = 0; c < span / 128; ++c) {
    const int64_t k0 = sp * span + c * 128;
    const float4 v = *reinterpret_cast<const float4*>(w + row * k + k0 + 4 * lane);
    const float x[4] = {v.x, v.y, v.z, v.w};
    uint32_t nib[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = s == 0.f ? 0 : __float2int_rn(rintf(__fdiv_rn(x[i], s)));
      const int qi = has_zero ? min(max(r + z, 0), 15) : min(max(r, -8), 7);
      nib[i] = static_cast<uint32_t>(qi) & 0xFu;
    }
    const uint16_t packed = static_cast<uint16_t>(nib[0] | (nib[1] << 4) | (nib[2] << 8) | (nib[3] << 12));
    *reinterpret_cast<uint16_t*>(q + row * (k / 2) + k0 / 2 + 2 * lane) = packed;
  }
  if ((4 * lane) % (group < 128 ? group : 128) == 0) scales[row * groups + gi] = sb;
}

// INT8, one warp per (row, group of 128); lane holds 4 consecutive K: s = bf16(fp32(amax)/127),
// q = clamp(rne(fp32(w/s)) [+ z]) into [-128, 127] (or [0, 255] with a u8 zero-point), one byte each.
__global__ void quant_int8_kernel(const float* __restrict__ w, const uint8_t* __restrict__ zeros, int64_t n,
                                  int64_t k, int has_zero, uint8_t* __restrict__ q, __nv_bfloat16* __restrict__ scales) {
  const int64_t groups = k / 128;
  const int64_t gid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gid >= n * groups) return;
  const int64_t row = gid / groups, g = gid % groups;
  const float4 v = *reinterpret_cast<const float4*>(w + row * k + g * 128 + 4 * lane);
  float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  amax = warp_max(amax, 32);
  const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(amax, 127.0f));
  const float s = __bfloat162float(sb);
  const int z = has_zero ? zeros[row * groups + g] : 0;
  const float x[4] = {v.x, v.y, v.z, v.w};
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = s == 0.f ? 0 : __float2int_rn(rintf(__fdiv_rn(x[i], s)));
    const int qi = has_zero ? min(max(r + z, 0), 255) : min(max(r, -128), 127);
    packed |= (static_cast<uint32_t>(qi) & 0xFFu) << (8 * i);
  }
  *reinterpret_cast<uint32_t*>(q + row * k + g * 128 + 4 * lane) = packed;
  if (lane == 0) scales[row * groups + g] = sb;
}

// MXFP4, one warp per (row, 128 K); 8 lanes per 32-block.
__global__ void quant_mx_kernel(const float* __restrict__ w, int64_t n, int64_t k,
                                uint8_t* __restrict__ q, uint8_t* __restrict__ e8) {
  const int64_t chunks = k / 128;
  const int64_t gid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gid >= n * chunks) return;
  const int64_t row = gid / chunks, c = gid % chunks;
  const float4 v = *reinterpret_cast<const float4*>(w + row * k + c * 128 + 4 * lane);
  float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  const int be = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  const int code = amax == 0.f ? 0 : min(max(be - 2, 0), 254);
  const float mul = pow2f(127 - code);
  const uint32_t b0 = e2m1x2(__fmul_rn(v.x, mul), __fmul_rn(v.y, mul));
  const uint32_t b1 = e2m1x2(__fmul_rn(v.z, mul), __fmul_rn(v.w, mul));
  *reinterpret_cast<uint16_t*>(q + row * (k / 2) + c * 64 + 2 * lane) = static_cast<uint16_t>(b0 | (b1 << 8));
  if ((lane & 7) == 0) e8[row * (k / 32) + c * 4 + (lane >> 3)] = static_cast<uint8_t>(code);
}

// MXINT4, one warp per (row, 128 K); 8 lanes per 32-block. Shared exponent as for MXFP4
// (floor(log2 amax) - 2, 2 being the largest power of two in the int4 range), elements
// clamp(RNE(w / 2^(e-127)), -8, 7) stored as two's-complement nibbles, even K in the low nibble.
__global__ void quant_mxint_kernel(const float* __restrict__ w, int64_t n, int64_t k,
                                   uint8_t* __restrict__ q, uint8_t* __restrict__ e8) {
  const int64_t chunks = k / 128;
  const int64_t gid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gid >= n * chunks) return;
  const int64_t row = gid / chunks, c = gid % chunks;
  const float4 v = *reinterpret_cast<const float4*>(w + row * k + c * 128 + 4 * lane);
  float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  const int be = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  const int code = amax == 0.f ? 0 : min(max(be - 2, 0), 254);
  const float mul = pow2f(127 - code);   // exact: a power of two, |w * mul| < 8
  const float x[4] = {v.x, v.y, v.z, v.w};
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int qi = min(max(__float2int_rn(__fmul_rn(x[i], mul)), -8), 7);
    packed |= (static_cast<uint32_t>(qi) & 0xFu) << (4 * i);
  }
  *reinterpret_cast<uint16_t*>(q + row * (k / 2) + c * 64 + 2 * lane) = static_cast<uint16_t>(packed);
  if ((lane & 7) == 0) e8[row * (k / 32) + c * 4 + (lane >> 3)] = static_cast<uint8_t>(code);
}

// Max |x| over a float array into per-block partials.
__global__ void amax_f32_kernel(const float* __restrict__ x, int64_t count, float* __restrict__ partial) {
  float m = 0.f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    m = fmaxf(m, fabsf(x[i]));
  m = warp_max(m, 32);
  __shared__ float red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.f;
    m = warp_max(m, 32);
    if (threadIdx.x == 0) partial[blockIdx.x] = m;
  }
}

__device__ __forceinline__ float reduce_partials(const float* partial, int count) {
  __shared__ float red[32];
  float m = 0.f;
  for (int i = threadIdx.x; i < count; i += blockDim.x) m = fmaxf(m, partial[i]);
  m = warp_max(m, 32);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x / 32); ++i) m = fmaxf(m, red[i]);
  return m;
}

constexpr int kAmaxBlocks = 512;

// NVFP4 weights: 4 lanes per 16-block; the tensor amax comes from the partials.
__global__ void quant_nv_kernel(const float* __restrict__ w, int64_t n, int64_t k,
                                const float* __restrict__ partial, int nparts, uint8_t* __restrict__ q,
                                uint8_t* __restrict__ sbo, float* __restrict__ g_out) {
  const float amax = reduce_partials(partial, nparts);
  const float g = amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  const int64_t quad = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // 4 elements
  const bool valid = quad < n * k / 4;  // k % 16 == 0: a 16-block never straddles the end
  const float4 v = valid ? *reinterpret_cast<const float4*>(w + quad * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  float bmax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));
  bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 2));
  if (!valid) return;
  const uint32_t sb = e4m3_code(__fdiv_rn(__fdiv_rn(bmax, 6.0f), g));
  const float denom = __fmul_rn(e4m3_value(sb), g);
  float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = denom > 0.f ? __fdiv_rn(x[i], denom) : 0.f;
  const uint32_t b0 = e2m1x2(x[0], x[1]), b1 = e2m1x2(x[2], x[3]);
  *reinterpret_cast<uint16_t*>(q + quad * 2) = static_cast<uint16_t>(b0 | (b1 << 8));
  if ((threadIdx.x & 3) == 0) sbo[quad / 4] = static_cast<uint8_t>(sb);
}

// ------------------------------------------------------------------ transform

__device__ void write_header(uint8_t* packed, int32_t fmt, int64_t n, int64_t k, int32_t has_zero,
                             float gw) {
  // called by 64 threads of one block: zero the 256 bytes, then thread 0 fills the fields
  reinterpret_cast<uint32_t*>(packed)[threadIdx.x] = 0u;
  __syncwarp();
  __threadfence_block();
  if (threadIdx.x == 0) {
    PackedHeader h;
    h.magic = kMagic;
    h.fmt = static_cast<uint32_t>(fmt);
    h.n = n;
    h.k = k;
    h.n_pad = (n + 127) / 128 * 128;
    h.k_pad = fmt == kW4A4Nv ? (k + 255) / 256 * 256 : k;
    h.has_zero = static_cast<uint32_t>(has_zero);
    h.tensor_scale = gw;
    const int64_t np = h.n_pad, kp = h.k_pad;
    if (unit_fmt(fmt))
      h.payload_bytes = static_cast<uint64_t>(np / 128) * (kp / 128) * unit_bytes(fmt, has_zero != 0);
    else
      h.payload_bytes = static_cast<uint64_t>(np) * kp / 2 +
                        static_cast<uint64_t>(np / 128) * (kp / (fmt == kW4A8Mx ? 128 : 64)) * kAtomBytes;
    *reinterpret_cast<PackedHeader*>(packed) = h;
  }
}

// Standard 32-bit word (byte i = columns 2i | 2i+1 << 4) -> unit word (even columns in the low
// half-word, odd in the high one).
__device__ __forceinline__ uint32_t interleave_word(uint32_t s) {
  uint32_t lo = s & 0x0F0F0F0Fu;
  uint32_t hi = (s >> 4) & 0x0F0F0F0Fu;
  lo = (lo | (lo >> 4)) & 0x00FF00FFu;
  lo = (lo | (lo >> 8)) & 0x0000FFFFu;
  hi = (hi | (hi >> 4)) & 0x00FF00FFu;
  hi = (hi | (hi >> 8)) & 0x0000FFFFu;
  return lo | (hi << 16);
}

// Zero-point as the packed weight holds it, from the standard-format value in `conv` (0: z itself;
// 1: (z - 1) mod 16, GPTQ-style).
__device__ __forceinline__ uint32_t zero_point(uint8_t stored, int32_t conv) {
  const uint32_t v = stored & 0xFu;
  return conv == 1 ? ((v + 1u) & 0xFu) : v;
}

// One block (128 threads, thread = row) per 128x128 unit. INT4 scales (and zero-points) come in
// groups of `group` along K: a group of 128 j gives every unit of its j k-blocks its scale; groups
// of 32 / 64 (format 6) give each 32-K chunk of a unit its own.
__global__ void transform_units_kernel(int32_t fmt, int32_t has_zero, int64_t n, int64_t k, int64_t group,
                                       int32_t zconv, const uint8_t* __restrict__ q, const void* __restrict__ scales,
                                       const uint8_t* __restrict__ zeros, uint8_t* __restrict__ packed) {
  const int64_t kbt = k / 128;
  const int64_t nt = blockIdx.x / kbt, kb = blockIdx.x % kbt;
  const int r = threadIdx.x;
  const int64_t row = nt * 128 + r;
  const uint32_t ub = unit_bytes(fmt, has_zero != 0);
  uint8_t* unit = packed + kHeaderBytes + static_cast<size_t>(blockIdx.x) * ub;
  if (blockIdx.x == 0 && threadIdx.x < 64) write_header(packed, fmt, n, k, has_zero, 1.0f);
  const bool valid = row < n;
  if (fmt == kW8A16Int8) {
    // one byte per code: the row's 128 codes in 16-column chunks, 2048 bytes apart (signed codes
    // stored as q + 128 = q ^ 0x80)
    const uint32_t flip8 = has_zero ? 0u : 0x80808080u;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (valid) {
        v = *reinterpret_cast<const uint4*>(q + row * k + kb * 128 + c * 16);
        v.x ^= flip8; v.y ^= flip8; v.z ^= flip8; v.w ^= flip8;
      }
      *reinterpret_cast<uint4*>(unit + c * 2048 + r * 16) = v;
    }
    uint16_t sb = 0;
    if (valid) sb = reinterpret_cast<const uint16_t*>(scales)[row * kbt + kb];
    *reinterpret_cast<uint16_t*>(unit + kUnitInt8Codes + 2 * r) = sb;
    if (has_zero) unit[kUnitInt8 + r] = valid ? zeros[row * kbt + kb] : 0;
    return;
  }
  // signed nibbles (INT4 without zero-points, MXINT4) are stored as q + 8 = q ^ 8
  const bool int4 = fmt == kW4A16Int4 || fmt == kW4A16Int4G;
  const uint32_t flip = ((int4 && !has_zero) || fmt == kW4A16MxInt) ? 0x88888888u : 0u;
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    uint4 src = make_uint4(0, 0, 0, 0);
    if (valid) src = *reinterpret_cast<const uint4*>(q + row * (k / 2) + kb * 64 + c4 * 16);
    uint4 dst;
    dst.x = valid ? interleave_word(src.x ^ flip) : 0u;
    dst.y = valid ? interleave_word(src.y ^ flip) : 0u;
    dst.z = valid ? interleave_word(src.z ^ flip) : 0u;
    dst.w = valid ? interleave_word(src.w ^ flip) : 0u;
    *reinterpret_cast<uint4*>(unit + c4 * 2048 + r * 16) = dst;
  }
  if (e8_unit_fmt(fmt)) {
    uint32_t e4 = 0;
    if (valid) e4 = *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(scales) + row * (k / 32) + kb * 4);
    *reinterpret_cast<uint32_t*>(unit + kUnitCodes + 4 * r) = e4;
  } else if (fmt == kW4A16Int4G) {
    const int64_t groups = k / group;
    uint16_t sb[4] = {0, 0, 0, 0};
    uint32_t z[4] = {0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int64_t gi = (kb * 128 + 32 * c) / group;
      if (valid) {
        sb[c] = reinterpret_cast<const uint16_t*>(scales)[row * groups + gi];
        if (has_zero) z[c] = zero_point(zeros[row * groups + gi], zconv);
      }
    }
    *reinterpret_cast<uint2*>(unit + kUnitCodes + 8 * r) =
        make_uint2(sb[0] | (static_cast<uint32_t>(sb[1]) << 16), sb[2] | (static_cast<uint32_t>(sb[3]) << 16));
    if (has_zero)
      *reinterpret_cast<uint16_t*>(unit + kUnitG32 + 2 * r) =
          static_cast<uint16_t>(z[0] | (z[1] << 4) | (z[2] << 8) | (z[3] << 12));
  } else {
    const int64_t groups = k / group, gi = (kb * 128) / group;
    uint16_t sb = 0;
    if (valid) sb = reinterpret_cast<const uint16_t*>(scales)[row * groups + gi];
    *reinterpret_cast<uint16_t*>(unit + kUnitCodes + 2 * r) = sb;
    if (has_zero) {
      uint32_t z = valid ? zero_point(zeros[row * groups + gi], zconv) : 0u;
      const uint32_t z_next = __shfl_down_sync(0xffffffffu, z, 1);
      if ((r & 1) == 0) unit[kUnitInt4 + r / 2] = static_cast<uint8_t>(z | (z_next << 4));
    }
  }
}

// Row-major codes with zero padding to [n_pad][k_pad/2]; 16 bytes per thread.
__global__ void transform_codes_kernel(int64_t n, int64_t k, int64_t n_pad, int64_t k_pad,
                                       const uint8_t* __restrict__ q, uint8_t* __restrict__ dst) {
  const int64_t per_row = k_pad / 32;  // 16-byte chunks per padded row
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_pad * per_row) return;
  const int64_t row = i / per_row, col = (i % per_row) * 16;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (row < n && col < k / 2) v = *reinterpret_cast<const uint4*>(q + row * (k / 2) + col);
  *reinterpret_cast<uint4*>(dst + row * (k_pad / 2) + col) = v;
}

// Scale-factor atoms: one thread per (row, chunk) writes its 4 scales.
__global__ void transform_atoms_kernel(int64_t n, int64_t n_pad, int64_t chunks_real, int64_t chunks_pad,
                                       const uint8_t* __restrict__ sf, uint8_t* __restrict__ atoms) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_pad * chunks_pad) return;
  const int64_t row = i % n_pad;
  const int64_t ch = i / n_pad;
  uint32_t v = 0;
  if (row < n && ch < chunks_real) v = *reinterpret_cast<const uint32_t*>(sf + row * chunks_real * 4 + ch * 4);
  const int64_t nt = row / 128;
  const int r = static_cast<int>(row % 128);
  uint8_t* atom = atoms + (nt * chunks_pad + ch) * kAtomBytes;
  *reinterpret_cast<uint32_t*>(atom + (r % 32) * 16 + (r / 32) * 4) = v;
}

__global__ void header_kernel(uint8_t* packed, int32_t fmt, int64_t n, int64_t k, int32_t has_zero, float gw) {
  write_header(packed, fmt, n, k, has_zero, gw);
}

// ------------------------------------------------------------------ dequant test hook

__global__ void dequant_units_kernel(int32_t fmt, int32_t has_zero, int64_t n, int64_t k,
                                     const uint8_t* __restrict__ packed, __nv_bfloat16* __restrict__ w) {
  __shared__ float lut[16];
  if (threadIdx.x < 16) lut[threadIdx.x] = e2m1_value(threadIdx.x);
  __syncthreads();
  const int64_t kbt = k / 128;
  const int64_t nt = blockIdx.x / kbt, kb = blockIdx.x % kbt;
  const int r = threadIdx.x;
  const int64_t row = nt * 128 + r;
  if (row >= n) return;
  const uint32_t ub = unit_bytes(fmt, has_zero != 0);
  const uint8_t* unit = packed + kHeaderBytes + static_cast<size_t>(blockIdx.x) * ub;
  if (fmt == kW8A16Int8) {
    const __nv_bfloat162 s8 = bf16_pair(*reinterpret_cast<const uint16_t*>(unit + kUnitInt8Codes + 2 * r));
    const float zf = 8388608.0f + static_cast<float>(has_zero ? unit[kUnitInt8 + r] : 128u);
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(unit + c * 2048 + r * 16);
      const uint32_t words[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t p2[2];
        dq_int8_word(words[j], zf, s8, p2);
        o[2 * j] = p2[0];
        o[2 * j + 1] = p2[1];
      }
      uint4* dst = reinterpret_cast<uint4*>(w + row * k + kb * 128 + c * 16);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    return;
  }
  __nv_bfloat162 zz = int4_zero_pair(8), ss = bf16_pair(0);
  uint32_t e4 = 0;
  uint2 s4 = make_uint2(0u, 0u);   // format 6: bf16 scales of the four 32-K chunks
  uint32_t z4 = 0x8888u;           // format 6: their zero-points
  if (e8_unit_fmt(fmt)) {
    e4 = *reinterpret_cast<const uint32_t*>(unit + kUnitCodes + 4 * r);
  } else if (fmt == kW4A16Int4G) {
    s4 = *reinterpret_cast<const uint2*>(unit + kUnitCodes + 8 * r);
    if (has_zero) z4 = *reinterpret_cast<const uint16_t*>(unit + kUnitG32 + 2 * r);
  } else {
    ss = bf16_pair(*reinterpret_cast<const uint16_t*>(unit + kUnitCodes + 2 * r));
    if (has_zero) zz = int4_zero_pair((unit[kUnitInt4 + r / 2] >> (4 * (r & 1))) & 0xFu);
  }
  for (int c4 = 0; c4 < 4; ++c4) {
    const uint4 c = *reinterpret_cast<const uint4*>(unit + c4 * 2048 + r * 16);
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
    const uint32_t ex = (e4 >> (8 * c4)) & 0xFFu;
    const float scale = pow2f(static_cast<int>(ex) - 127);
    const __nv_bfloat162 si = bits_bf16x2(mxint_scale_pair(ex));
    if (fmt == kW4A16Int4G) {
      const uint32_t sw = c4 < 2 ? s4.x : s4.y;
      ss = bf16_pair(static_cast<uint16_t>(sw >> (16 * (c4 & 1))));
      zz = int4_zero_pair((z4 >> (4 * c4)) & 0xFu);
    }
    for (int j = 0; j < 4; ++j) {
      uint32_t o[4];
      if (fmt == kW4A16Mx) dq_mx_word(words[j], lut, scale, o);
      else if (fmt == kW4A16MxInt) dq_int4_word(words[j], zz, si, o);
      else dq_int4_word(words[j], zz, ss, o);
      *reinterpret_cast<uint4*>(w + row * k + kb * 128 + (4 * c4 + j) * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Row-major formats: thread per (row, 8 consecutive K).
__global__ void dequant_rowmajor_kernel(int32_t fmt, int64_t n, int64_t k, int64_t k_pad,
                                        const uint8_t* __restrict__ codes, const uint8_t* __restrict__ atoms,
                                        __nv_bfloat16* __restrict__ w) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n * (k / 8)) return;
  const int64_t row = i / (k / 8), k0 = (i % (k / 8)) * 8;
  const uint32_t c = *reinterpret_cast<const uint32_t*>(codes + row * (k_pad / 2) + k0 / 2);
  const int chunk_k = fmt == kW4A8Mx ? 128 : 64;
  const int64_t chunks_pad = k_pad / chunk_k;
  const int64_t ch = k0 / chunk_k;
  const int j = static_cast<int>((k0 % chunk_k) / (chunk_k / 4));
  const int r = static_cast<int>(row % 128);
  const uint8_t sfc = atoms[((row / 128) * chunks_pad + ch) * kAtomBytes + (r % 32) * 16 + (r / 32) * 4 + j];
  const float scale = fmt == kW4A8Mx ? pow2f(static_cast<int>(sfc) - 127) : e4m3_value(sfc);
  uint32_t o[4];
  for (int t = 0; t < 4; ++t) {
    const float lo = e2m1_value((c >> (8 * t)) & 0xFu) * scale;
    const float hi = e2m1_value((c >> (8 * t + 4)) & 0xFu) * scale;
    o[t] = pack_bf16x2_rn(lo, hi);
  }
  *reinterpret_cast<uint4*>(w + row * k + k0) = make_uint4(o[0], o[1], o[2], o[3]);
}

inline unsigned blocks_for(int64_t threads, int per_block) {
  return static_cast<unsigned>((threads + per_block - 1) / per_block);
}

}  // namespace

cudaError_t launch_quantize_weight(int32_t fmt, int32_t has_zero, int64_t n, int64_t k, int64_t group,
                                   const float* w, const uint8_t* zeros_in, uint8_t* q_out, void* scales_out,
                                   float* g_out, float* ws, cudaStream_t st) {
  if (fmt == kW8A16Int8) {
    quant_int8_kernel<<<blocks_for(n * (k / 128) * 32, 256), 256, 0, st>>>(
        w, zeros_in, n, k, has_zero, q_out, static_cast<__nv_bfloat16*>(scales_out));
  } else if (fmt == kW4A16Int4 || fmt == kW4A16Int4G) {
    const int64_t span = group < 128 ? 128 : group;
    quant_int4_kernel<<<blocks_for(n * (k / span) * 32, 256), 256, 0, st>>>(
        w, zeros_in, n, k, has_zero, group, q_out, static_cast<__nv_bfloat16*>(scales_out));
  } else if (fmt == kW4A16Mx || fmt == kW4A8Mx) {
    quant_mx_kernel<<<blocks_for(n * (k / 128) * 32, 256), 256, 0, st>>>(
        w, n, k, q_out, static_cast<uint8_t*>(scales_out));
  } else if (fmt == kW4A16MxInt) {
    quant_mxint_kernel<<<blocks_for(n * (k / 128) * 32, 256), 256, 0, st>>>(
        w, n, k, q_out, static_cast<uint8_t*>(scales_out));
  } else {
    amax_f32_kernel<<<kAmaxBlocks, 256, 0, st>>>(w, n * k, ws);
    quant_nv_kernel<<<blocks_for(n * k / 4, 256), 256, 0, st>>>(
        w, n, k, ws, kAmaxBlocks, q_out, static_cast<uint8_t*>(scales_out), g_out);
  }
  return cudaGetLastError();
}

size_t quantize_ws_floats() { return kAmaxBlocks; }

cudaError_t launch_transform(int32_t fmt, int32_t has_zero, int64_t n, int64_t k, float gw, int64_t group,
                             int32_t zconv, const uint8_t* q, const void* scales, const uint8_t* zeros,
                             uint8_t* packed, cudaStream_t st) {
  const int64_t n_pad = (n + 127) / 128 * 128;
  if (unit_fmt(fmt)) {
    transform_units_kernel<<<static_cast<unsigned>((n_pad / 128) * (k / 128)), 128, 0, st>>>(
        fmt, has_zero, n, k, group, zconv, q, scales, zeros, packed);
    return cudaGetLastError();
  }
  const int64_t k_pad = fmt == kW4A4Nv ? (k + 255) / 256 * 256 : k;
  header_kernel<<<1, 64, 0, st>>>(packed, fmt, n, k, 0, fmt == kW4A4Nv ? gw : 1.0f);
  uint8_t* body = packed + kHeaderBytes;
  transform_codes_kernel<<<blocks_for(n_pad * (k_pad / 32), 256), 256, 0, st>>>(n, k, n_pad, k_pad, q, body);
  const int chunk_k = fmt == kW4A8Mx ? 128 : 64;
  uint8_t* atoms = body + n_pad * k_pad / 2;
  transform_atoms_kernel<<<blocks_for(n_pad * (k_pad / chunk_k), 256), 256, 0, st>>>(
      n, n_pad, k / chunk_k, k_pad / chunk_k, static_cast<const uint8_t*>(scales), atoms);
  return cudaGetLastError();
}

cudaError_t launch_dequant(int32_t fmt, int32_t has_zero, int64_t n, int64_t k, const uint8_t* packed,
                           __nv_bfloat16* w, cudaStream_t st) {
  const int64_t n_pad = (n + 127) / 128 * 128;
  if (unit_fmt(fmt)) {
    dequant_units_kernel<<<static_cast<unsigned>((n_pad / 128) * (k / 128)), 128, 0, st>>>(
        fmt, has_zero, n, k, packed, w);
    return cudaGetLastError();
  }
  const int64_t k_pad = fmt == kW4A4Nv ? (k + 255) / 256 * 256 : k;
  const uint8_t* body = packed + kHeaderBytes;
  dequant_rowmajor_kernel<<<blocks_for(n * (k / 8), 256), 256, 0, st>>>(fmt, n, k, k_pad, body,
                                                                        body + n_pad * k_pad / 2, w);
  return cudaGetLastError();
}

}  // namespace hm
