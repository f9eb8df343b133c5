// Restoring 4-bit (and 8-bit) weight codes to bf16 in registers. Shared by the W4A16 GEMM's
// dequant warps and the hm_dequant test hook, so both restore exactly the same values.
//
// INT4 (the explainer page's rule, restored weight = scale * code, with an optional
// zero-point): w = bf16((u - z) * s). u and z are 4-bit unsigned; the pair (128 + u) is
// formed directly as bf16 bits (0x4300 = 128.0, whose last mantissa bit weighs 1, so the
// nibble lands in the mantissa exactly), (128 + u) - (128 + z) is exact in bf16, and the
// product with the bf16 scale is rounded once (round-to-nearest-even), as the definition asks.
//
// MXFP4 (OCP MX v1.0): w = e2m1(code) * 2^(e-127), formed in fp32 (exact) and converted to
// bf16 with round-to-nearest-even (exact in the normal range).
//
// MXINT4 (signed 4-bit integers q in [-8, 7] with an E8M0 scale per 32): w = q * 2^(e-127).
// Units hold u = q + 8, so the INT4 restore with z = 8 gives q exactly and one bf16 multiply
// by 2^(e-127) scales it; q has at most four significant bits, so that product is exact.
#pragma once
#include <cuda_bf16.h>

#include "hm_device.cuh"

namespace hm {

// One 32-bit word of the unit layout -> 8 consecutive bf16 (as 4 bf16x2 registers). Written as
// explicit PTX so that each pair costs one shift, one lop3 (mask | magic), one bf16x2 subtract
// (exact: both operands are integers in [128, 143]) and one bf16x2 multiply (one rounding).
__device__ __forceinline__ void dq_int4_word(uint32_t w, __nv_bfloat162 zz, __nv_bfloat162 ss,
                                             uint32_t (&o)[4]) {
  const uint32_t z2 = bf16x2_bits(zz), s2 = bf16x2_bits(ss);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t t, v;
    const uint32_t sh = w >> (4 * i);
    asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(t) : "r"(sh));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(v) : "r"(t), "r"(z2));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(v), "r"(s2));
  }
}

// One word -> 8 consecutive bf16 holding u - z exactly (integers in [-15, 15]), for kernels
// that apply the group scale to the fp32 partial sum of the group instead of to each weight.
__device__ __forceinline__ void dq_int4_word_unscaled(uint32_t w, uint32_t z2, uint32_t (&o)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t t;
    const uint32_t sh = w >> (4 * i);
    asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(t) : "r"(sh));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(t), "r"(z2));
  }
}

// INT8: one 32-bit word of 4 codes (bytes, k order) -> 2 bf16x2 pairs holding u - z exactly
// (integers in [-255, 255] need at most 8 significant bits). Each byte goes into the low mantissa
// of the fp32 2^23 (a byte permute), the fp32 subtraction of 2^23 + z is exact, and the pair is
// packed to bf16 (exact). zf = 2^23 + z as fp32.
__device__ __forceinline__ void dq_int8_word_unscaled(uint32_t w, float zf, uint32_t (&o)[2]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(w), "r"(0x4B000000u), "r"(0x7540u | (2u * i)));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b) : "r"(w), "r"(0x4B000000u), "r"(0x7540u | (2u * i + 1u)));
    o[i] = pack_bf16x2_rn(__uint_as_float(a) - zf, __uint_as_float(b) - zf);
  }
}

// INT8 word -> 2 bf16x2 pairs of the restored weight bf16((u - z) * s): the exact pairs above times
// the bf16 scale, rounded once.
__device__ __forceinline__ void dq_int8_word(uint32_t w, float zf, __nv_bfloat162 ss, uint32_t (&o)[2]) {
  uint32_t e[2];
  dq_int8_word_unscaled(w, zf, e);
  const uint32_t s2 = bf16x2_bits(ss);
#pragma unroll
  for (int i = 0; i < 2; ++i) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(e[i]), "r"(s2));
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

// MXFP4 restore without a table. The three magnitude bits of an e2m1 code (exponent e1 e0,
// mantissa m) placed at bf16 bits [8:6], with the sign at bit 15, form the bf16 number
// code * 2^-126: codes with e = 0 land on bf16 subnormals (m * 2^-127), the others on normals
// 2^(e-127) * (1 + m/2). One bf16 multiply by 2^(E-1) then gives code * 2^(E-127) with a
// single rounding, the restored weight of the OCP MX definition. sc2 holds 2^(E-1) in both
// halves, which bf16 can represent for E <= 128; callers take dq_mx_word above otherwise.
// Nibble pairing is that of dq_mx_word: nibble i of w goes to the low half, nibble i + 4 to the
// high half of o[i].
__device__ __forceinline__ uint32_t mx_pow2_pair(uint32_t e) {
  return ((e + 126u) << 7) * 0x00010001u;
}

__device__ __forceinline__ void dq_mx_word_bits(uint32_t w, uint32_t sc2, uint32_t (&o)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t a = (6 - 4 * i) >= 0 ? (w << (6 - 4 * i)) : (w >> (4 * i - 6));
    const uint32_t b = w << (12 - 4 * i);
    uint32_t v;
    asm("lop3.b32 %0, %1, 0x01C001C0, %2, 0xEA;" : "=r"(v) : "r"(a), "r"(b & 0x80008000u));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(v), "r"(sc2));
  }
}

// bf16x2 holding 2^(e-127) in both halves, for an E8M0 code e: the normal 2^(e-127) for
// e = 1..254 (exponent field e, zero mantissa) and the subnormal 2^-127 for e = 0. The NaN code
// 255 gives infinity, so a block marked NaN restores to non-finite values.
__device__ __forceinline__ uint32_t mxint_scale_pair(uint32_t e) {
  const uint32_t b = e == 0u ? 0x0040u : (e << 7);
  return b * 0x00010001u;
}

}  // namespace hm
