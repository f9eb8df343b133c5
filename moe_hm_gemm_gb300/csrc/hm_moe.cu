// MoE token movement around the grouped GEMMs: the gather of each token's activation row into
// the expert-sorted order the grouped GEMM reads, and the weighted top-k combine of the expert
// outputs back into one row per token.
//
// The explainer page ("vLLM Humming은 4비트를 어떻게 계산하나", MoE paragraph of the section "같은
// 가중치도 한 토큰과 많은 토큰에서 비용이 다르다") routes every token to some experts, each expert
// multiplying only its own tokens; the pages do not print the two steps around that product, so
// the usual top-k layer is read:
//   gather:  xs[r][:] = x[token_of_row[r]][:]                        (an exact copy)
//   combine: out[t][:] = bf16( sum over slots j of w[t][j] * y[pos[t][j]][:] ), pos < 0 = empty
// The combine sums in fp32 with one fused multiply-add per slot, in slot order j = 0, 1, ..., so
// a call is deterministic; the one rounding into bf16 comes last.
//
// Both are HBM-bound streaming kernels: 8 bf16 columns (16 bytes) per thread and step,
// grid-stride over at most 8 CTAs of 256 threads per SM. Indices outside their range set bit 3 of
// the device error word; the row (gather) or slot (combine) is then treated as zeros.
#include <cuda_bf16.h>

#include "hm_device.cuh"
#include "hm_kernels.h"

namespace hm {
namespace {

constexpr uint32_t kErrBadIndex = 8u;   // device error bit 3

__device__ __forceinline__ void bf16x8_acc(uint4 v, float wgt, float (&acc)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = fmaf(wgt, __uint_as_float(u[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = fmaf(wgt, __uint_as_float(u[i] & 0xFFFF0000u), acc[2 * i + 1]);
  }
}

__global__ void __launch_bounds__(256) moe_gather_kernel(const __nv_bfloat16* __restrict__ x,
                                                         const int32_t* __restrict__ token_of_row,
                                                         __nv_bfloat16* __restrict__ xs, int64_t tokens,
                                                         int64_t rows, int64_t k, uint32_t* err) {
  const int64_t per_row = k / 8;
  const int64_t total = rows * per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row, c8 = i - r * per_row;
    const int64_t t = __ldg(token_of_row + r);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (t >= 0 && t < tokens) {
      v = __ldg(reinterpret_cast<const uint4*>(x + t * k) + c8);
    } else if (c8 == 0) {
      atomicOr(err, kErrBadIndex);
    }
    __stcs(reinterpret_cast<uint4*>(xs + r * k) + c8, v);
  }
}

__global__ void __launch_bounds__(256) moe_combine_kernel(const __nv_bfloat16* __restrict__ y,
                                                          const int32_t* __restrict__ pos,
                                                          const float* __restrict__ w,
                                                          __nv_bfloat16* __restrict__ out, int64_t tokens,
                                                          int32_t topk, int64_t rows, int64_t n, uint32_t* err) {
  const int64_t per_row = n / 8;
  const int64_t total = tokens * per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / per_row, c8 = i - t * per_row;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int32_t* pt = pos + t * topk;
    const float* wt = w + t * topk;
    // up to four slots' rows in flight at a time, summed in slot order
    for (int32_t j0 = 0; j0 < topk; j0 += 4) {
      uint4 v[4];
      float wj[4];
      bool ok[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int32_t j = j0 + u;
        ok[u] = false;
        if (j < topk) {
          const int64_t r = __ldg(pt + j);
          ok[u] = r >= 0 && r < rows;
          if (ok[u]) {
            v[u] = __ldcs(reinterpret_cast<const uint4*>(y + r * n) + c8);
            wj[u] = __ldg(wt + j);
          } else if (r >= rows && c8 == 0) {
            atomicOr(err, kErrBadIndex);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (ok[u]) bf16x8_acc(v[u], wj[u], acc);
    }
    __stcs(reinterpret_cast<uint4*>(out + t * n) + c8,
           make_uint4(pack_bf16x2_rn(acc[0], acc[1]), pack_bf16x2_rn(acc[2], acc[3]),
                      pack_bf16x2_rn(acc[4], acc[5]), pack_bf16x2_rn(acc[6], acc[7])));
  }
}

unsigned grid_for(int64_t work, int num_sms) {
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  return static_cast<unsigned>(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_moe_gather(const __nv_bfloat16* x, const int32_t* token_of_row, __nv_bfloat16* xs,
                              int64_t tokens, int64_t rows, int64_t k, uint32_t* err, int num_sms,
                              cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  moe_gather_kernel<<<grid_for(rows * (k / 8), num_sms), 256, 0, st>>>(x, token_of_row, xs, tokens, rows, k, err);
  return cudaGetLastError();
}

cudaError_t launch_moe_combine(const __nv_bfloat16* y, const int32_t* pos, const float* w, __nv_bfloat16* out,
                               int64_t tokens, int32_t topk, int64_t rows, int64_t n, uint32_t* err, int num_sms,
                               cudaStream_t st) {
  if (tokens == 0) return cudaSuccess;
  moe_combine_kernel<<<grid_for(tokens * (n / 8), num_sms), 256, 0, st>>>(y, pos, w, out, tokens, topk, rows, n,
                                                                           err);
  return cudaGetLastError();
}

}  // namespace hm
