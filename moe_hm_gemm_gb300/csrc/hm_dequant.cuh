// Restoring 4-bit weight codes to bf16 in registers. Shared by the W4A16 GEMM's dequant
// warps and the hm_dequant test hook, so both restore exactly the same values.
//
// INT4 (the explainer page's rule, restored weight = scale * code, with an optional
// zero-point): w = bf16((u - z) * s). u and z are 4-bit unsigned; the pair (128 + u) is
// formed directly as bf16 bits (0x4300 = 128.0, whose last mantissa bit weighs 1, so the
// nibble lands in the mantissa exactly), (128 + u) - (128 + z) is exact in bf16, and the
// product with the bf16 scale is rounded once (round-to-nearest-even), as the definition asks.
//
// MXFP4 (OCP MX v1.0): w = e2m1(code) * 2^(e-127), formed in fp32 (exact) and converted to
// bf16 with round-to-nearest-even (exact in the normal range).
#pragma once
#include <cuda_bf16.h>

#include "hm_device.cuh"

namespace hm {

// One 32-bit word of the unit layout -> 8 consecutive bf16 (as 4 bf16x2 registers).
__device__ __forceinline__ void dq_int4_word(uint32_t w, __nv_bfloat162 zz, __nv_bfloat162 ss,
                                             uint32_t (&o)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
    const __nv_bfloat162 v = __hsub2(bits_bf16x2(t), zz);
    o[i] = bf16x2_bits(__hmul2(v, ss));
  }
}

// bf16x2 holding (128 + z, 128 + z).
__device__ __forceinline__ __nv_bfloat162 int4_zero_pair(uint32_t z) {
  const uint32_t b = 0x4300u | (z & 0xFu);
  return bits_bf16x2(b | (b << 16));
}

__device__ __forceinline__ __nv_bfloat162 bf16_pair(uint16_t bits) {
  return bits_bf16x2(static_cast<uint32_t>(bits) | (static_cast<uint32_t>(bits) << 16));
}

// e2m1 code -> value (fp32), from the bit fields: sign, 2 exponent bits (bias 1), 1 mantissa bit.
__host__ __device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t mag = c & 7u;
  // twice the magnitude: 0,1,2,3,4,6,8,12
  const uint32_t twice = mag < 2u ? mag : ((2u | (mag & 1u)) << ((mag >> 1) - 1u));
  const float v = 0.5f * static_cast<float>(twice);
  return (c & 8u) ? -v : v;
}

// 2^k as fp32 for k in [-149, 127] (subnormal results included).
__device__ __forceinline__ float pow2f(int k) {
  return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

// MXFP4 word -> 8 consecutive bf16. lut: e2m1 values (16 floats, shared memory); scale = 2^(e-127).
__device__ __forceinline__ void dq_mx_word(uint32_t w, const float* lut, float scale,
                                           uint32_t (&o)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = lut[(w >> (4 * i)) & 0xFu] * scale;
    const float hi = lut[(w >> (16 + 4 * i)) & 0xFu] * scale;
    o[i] = pack_bf16x2_rn(lo, hi);
  }
}

}  // namespace hm
