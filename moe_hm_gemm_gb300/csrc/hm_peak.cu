// Tensor-core throughput probe: the dense peak of each tcgen05 MMA kind this library issues,
// measured on the device that runs the GEMMs, so that the tensor-bound roofline of each format is
// taken against a measured peak of its own MMA kind.
//
// One CTA per SM; every operand sits in shared memory (filled once, no loads in the loop) and the
// accumulators in TMEM. Several warps issue MMAs into accumulators of their own (one issuing
// thread waits ~50 cycles per instruction, which would otherwise cap the narrow kinds), each
// runs `iters` rounds of four MMAs over a 128-byte-wide K slice, commits once and waits (bounded)
// for its MMAs to complete. Shapes and kinds:
//   kind 0: kind::f16, bf16 x bf16, M = 128, N = 256, K = 16, two issuers;
//   kind 1: kind::mxf8f6f4.block_scale.scale_vec::1X, e4m3 x e4m3 with UE8M0 scales, M = N = 128,
//           K = 32, three issuers;
//   kind 2: kind::mxf4nvf4.block_scale.scale_vec::4X, e2m1 x e2m1 with UE4M3 scales, M = N = 128,
//           K = 64, three issuers;
//   kinds 3 and 4: kinds 1 and 2 with N = 256 and one issuer (the widest instruction of the kind);
//   kind 5: kind::f16 with M = 128, N = 256, K = 16, A read from TMEM, one issuer (the instruction
//           and issue pattern of the W4A16 kernel's 256-token tiles: what one issuing thread can
//           sustain); kind 6: the same with A in shared memory.
// The operand values are arbitrary finite numbers (the tensor pipe's rate does not depend on
// them). The caller times the launch with events; hm_mma_peak_probe reports the FLOPs it issued.
#include <cuda_bf16.h>

#include "hm_device.cuh"
#include "hm_kernels.h"

namespace hm {
namespace {

constexpr int kPeakThreads = 128;
constexpr int kPeakSmem = 120 * 1024;   // keeps one CTA per SM (the probe allocates all of TMEM)

template <int KIND>
struct PeakShape {
  static constexpr bool kF16 = KIND == 0 || KIND >= 5;                               // kind::f16
  static constexpr int kN = (KIND == 1 || KIND == 2) ? 128 : 256;
  static constexpr int kK = kF16 ? 16 : ((KIND == 1 || KIND == 3) ? 32 : 64);         // K per instruction
  static constexpr int kIssuers = KIND == 0 ? 2 : (KIND >= 3 ? 1 : 3);
  static constexpr int kATmemCol = 256;                                               // kind 5: A in TMEM
  static constexpr int kSfCol = KIND >= 3 ? 256 : 384;                               // first scale column
  static constexpr int kAOff = 0;                                     // 128 rows x 128 bytes
  static constexpr int kBOff = 128 * 128;                             // kN rows x 128 bytes
  static constexpr int kSfOff = kBOff + kN * 128;                     // 8 scale atoms of 512 bytes
  static constexpr int kBarOff = kSfOff + 8 * 512;
  static constexpr int kEnd = kBarOff + 64;
  static_assert(kEnd + 1024 <= kPeakSmem, "shared memory");
};

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7FEB352Du;
  x ^= x >> 15;
  x *= 0x846CA68Bu;
  x ^= x >> 16;
  return x;
}

template <int KIND>
__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(int32_t iters, uint32_t* err, uint64_t timeout_ns) {
  using S = PeakShape<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* done = reinterpret_cast<uint64_t*>(smem + S::kBarOff);   // [issuer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kBarOff + 32);
  const int warp = threadIdx.x >> 5;

  // operands: arbitrary finite values of each type
  uint32_t* words = reinterpret_cast<uint32_t*>(smem);
  for (int i = threadIdx.x; i < S::kSfOff / 4; i += kPeakThreads) {
    const uint32_t h = mix32(static_cast<uint32_t>(i) * 2654435761u + blockIdx.x);
    uint32_t v;
    if (S::kF16) {
      v = (h & 0x807F807Fu) | 0x3C003C00u;   // bf16 values of magnitude in [2^-7, 2^-6)
    } else if (KIND == 1 || KIND == 3) {
      v = h & 0xF7F7F7F7u;                   // e4m3 without the NaN codes (exponent field <= 14)
    } else {
      v = h;                                 // e2m1: every code is finite
    }
    words[i] = v;
  }
  // scale factors: 1.0 (UE8M0 127, UE4M3 0x38)
  const uint32_t one4 = (KIND == 1 || KIND == 3) ? 0x7F7F7F7Fu : 0x38383838u;
  for (int i = threadIdx.x; i < 8 * 512 / 4; i += kPeakThreads) words[S::kSfOff / 4 + i] = one4;
  if (threadIdx.x == 0) {
    for (int w = 0; w < S::kIssuers; ++w) mbar_init(&done[w], 1);
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (KIND == 5) {   // A in TMEM: every warp fills its 32 lanes of the 32 columns the 4 K-steps read
    uint32_t r[32];
    for (int i = 0; i < 32; ++i)
      r[i] = (mix32(static_cast<uint32_t>(i * 77 + threadIdx.x) + blockIdx.x) & 0x807F807Fu) | 0x3C003C00u;
    tmem_st32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + S::kATmemCol, r);
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  const int issuer = warp - 1;
  if (issuer >= 0 && issuer < S::kIssuers && (threadIdx.x & 31) == 0) {
    const uint32_t a0 = smem_u32(smem + S::kAOff), b0 = smem_u32(smem + S::kBOff);
    const uint32_t d = tmem + static_cast<uint32_t>(issuer * S::kN);
    // this issuer's scale-factor columns (block-scaled kinds): after the accumulators
    const uint32_t sf = tmem + static_cast<uint32_t>(S::kSfCol) + static_cast<uint32_t>(issuer * 32);
    // (kinds 3 and 4: the B scales of 256 rows span twice the columns of 128; all of them lie in
    // the allocation and hold 1.0)
    if (KIND == 1 || KIND == 3) {
      for (int j = 0; j < (KIND == 3 ? 4 : 2); ++j)
        tc_cp_32x128b_x4(sf + 4 * j, sdesc_sf(smem_u32(smem + S::kSfOff + 512 * j)));
    } else if (KIND == 2 || KIND == 4) {
      for (int j = 0; j < 8; ++j) tc_cp_32x128b_x4(sf + 4 * j, sdesc_sf(smem_u32(smem + S::kSfOff + 512 * j)));
      if (KIND == 4)
        for (int j = 0; j < 8; ++j) tc_cp_32x128b_x4(sf + 32 + 4 * j, sdesc_sf(smem_u32(smem + S::kSfOff + 512 * j)));
    }
    for (int32_t it = 0; it < iters; ++it) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = sdesc_sw128(a0 + 32 * k);
        const uint64_t bd = sdesc_sw128(b0 + 32 * k);
        const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
        if constexpr (KIND == 5) {
          mma_bf16_ta(d, tmem + S::kATmemCol + 8 * k, bd, idesc_bf16(128, S::kN), acc);
        } else if constexpr (S::kF16) {
          mma_bf16(d, ad, bd, idesc_bf16(128, S::kN), acc);
        } else if constexpr (KIND == 1 || KIND == 3) {
          mma_mxf8f6f4(d, ad, bd, idesc_block_scaled(128, S::kN, 0, 0, 1, k, k), sf, sf + 4, acc);
        } else {
          mma_mxf4nvf4_4x(d, ad, bd, idesc_block_scaled(128, S::kN, 1, 1, 0, 0, 0), sf + 4 * k,
                          sf + (KIND == 4 ? 32 + 8 * k : 16 + 4 * k), acc);
        }
      }
    }
    tc_commit(&done[issuer]);
    // bounded wait for this issuer's MMAs (and scale copies) to complete
    const uint32_t bar = smem_u32(&done[issuer]);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, 0)) {
      if (globaltimer() - t0 > timeout_ns) {
        atomicOr(err, kErrTimeout);
        break;
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int KIND>
cudaError_t launch_peak(int32_t iters, int num_sms, uint32_t* err, uint64_t timeout_ns, cudaStream_t st,
                        double* flops) {
  using S = PeakShape<KIND>;
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(mma_peak_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  *flops = static_cast<double>(num_sms) * iters * 4 * S::kIssuers * 2.0 * 128 * S::kN * S::kK;
  mma_peak_kernel<KIND><<<num_sms, kPeakThreads, kPeakSmem, st>>>(iters, err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mma_peak(int kind, int32_t iters, int num_sms, uint32_t* err, uint64_t timeout_ns,
                            cudaStream_t st, double* flops) {
  if (kind == 0) return launch_peak<0>(iters, num_sms, err, timeout_ns, st, flops);
  if (kind == 1) return launch_peak<1>(iters, num_sms, err, timeout_ns, st, flops);
  if (kind == 2) return launch_peak<2>(iters, num_sms, err, timeout_ns, st, flops);
  if (kind == 3) return launch_peak<3>(iters, num_sms, err, timeout_ns, st, flops);
  if (kind == 4) return launch_peak<4>(iters, num_sms, err, timeout_ns, st, flops);
  if (kind == 5) return launch_peak<5>(iters, num_sms, err, timeout_ns, st, flops);
  if (kind == 6) return launch_peak<6>(iters, num_sms, err, timeout_ns, st, flops);
  return cudaErrorInvalidValue;
}

}  // namespace hm
