// Activation quantizers (per call, on the hot path of the W4A8 and W4A4 GEMMs) and the
// bounded-wait probe.
//
// FP8 per token: the W4A8 path of the explainer page ("vLLM Humming은 4비트를 어떻게
// 계산하나", section "가중치 형식, 활성값, 백엔드를 한 줄에 적는다": activations go from BF16 to
// per-token FP8). Per row: amax; s_tok = fp32(amax/448); inv = fp32(448/amax);
// xq = e4m3(RNE, satfinite)(fp32(x*inv)); a zero row gives s_tok = 0, xq = 0.
//
// NVFP4 (named on the news page's format list): gX = fp32(amax/2688) (or the caller's),
// per 16 along K sb = e4m3(fp32(fp32(amax16/6)/gX)), element e2m1(fp32(x/fp32(sb*gX))).
// Both are HBM-bound streaming kernels: each input byte is read once (twice for the
// two-pass NVFP4 tensor scale) and the outputs are written once with 16-byte or 8-byte
// stores.
//
// MoE expert activation between the grouped GEMMs (the MoE layer of the explainer page, MoE
// paragraph of the section "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다"; the activation
// itself is not printed on the pages, the usual gated SiLU is taken): h = bf16(SiLU(gate) * up)
// with SiLU(v) = v / (1 + exp(-v)) in fp32 (evaluated as v * logistic(v) from exp(-|v|)), gate
// the first and up the second half of each gate-up row. Streaming: 8 columns per thread and step (two 16-byte loads, one 16-byte store).
#include <cuda_bf16.h>

#include "hm_dequant.cuh"
#include "hm_device.cuh"
#include "hm_kernels.h"
#include "hm_layout.h"

namespace hm {
namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u16.u8 %0, b;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float mag = e == 0 ? static_cast<float>(m) * 0.001953125f
                           : static_cast<float>(8u + m) * pow2f(static_cast<int>(e) - 10);
  return (c & 0x80u) ? -mag : mag;
}

__device__ __forceinline__ void bf16x8_to_f32(uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

constexpr int kFp8Threads = 256;

// One block per row.
__global__ void __launch_bounds__(kFp8Threads) act_fp8_kernel(const __nv_bfloat16* __restrict__ x, int64_t k,
                                                              uint8_t* __restrict__ xq, float* __restrict__ s_tok) {
  const int64_t row = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(x + row * k);
  const int64_t chunks = k / 8;
  float amax = 0.f;
  for (int64_t i = threadIdx.x; i < chunks; i += kFp8Threads) {
    float f[8];
    bf16x8_to_f32(__ldg(src + i), f);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
  }
  __shared__ float red[kFp8Threads / 32];
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.f;
#pragma unroll
  for (int i = 0; i < kFp8Threads / 32; ++i) amax = fmaxf(amax, red[i]);
  const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 0.f;
  if (threadIdx.x == 0) s_tok[row] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(xq + row * k);
  for (int64_t i = threadIdx.x; i < chunks; i += kFp8Threads) {
    float f[8];
    bf16x8_to_f32(__ldg(src + i), f);
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = e4m3x2(__fmul_rn(f[2 * j], inv), __fmul_rn(f[2 * j + 1], inv));
    dst[i] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
  }
}

constexpr int kAmaxBlocks = 512;

__global__ void amax_bf16_kernel(const __nv_bfloat16* __restrict__ x, int64_t count8, float* __restrict__ partial) {
  const uint4* src = reinterpret_cast<const uint4*>(x);
  float m = 0.f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float f[8];
    bf16x8_to_f32(__ldg(src + i), f);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
  }
  __shared__ float red[32];
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < static_cast<int>(blockDim.x / 32); ++i) t = fmaxf(t, red[i]);
    partial[blockIdx.x] = t;
  }
}

// MoE W4A4 activations: the scale atoms of expert-sorted rows are laid out per expert token tile
// (an expert's rows need not start on a 128-row boundary): row r of expert e (rows offs[e] ..
// offs[e+1]-1) is row i % bt of atom block tpre[e] + i / bt, i = r - offs[e], where tpre[e] is the
// number of token tiles of bt rows of the experts before e. row_slot[r] = block * 128 + row within
// the block, or -1 for a row of no expert (r >= offs[E]) or a block past `max_blocks`.
constexpr int kSlotMaxExperts = 1024;
__global__ void __launch_bounds__(1024) moe_row_slots_kernel(const int32_t* __restrict__ offsets, int E, int64_t rows,
                                                             int bt, int64_t max_blocks, int32_t* __restrict__ row_slot) {
  __shared__ int32_t offs[kSlotMaxExperts + 1];
  __shared__ int32_t tpre[kSlotMaxExperts + 1];
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        const int a = offsets[e], b = offsets[e + 1];
        offs[e] = a;
        local += b > a ? (b - a + bt - 1) / bt : 0;
      }
    }
    if (lane == 0) offs[E] = offsets[E];
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        tpre[e] = run;
        const int a = offsets[e], b = offsets[e + 1];
        run += b > a ? (b - a + bt - 1) / bt : 0;
      }
    }
  }
  __syncthreads();
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < rows;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int32_t slot = -1;
    if (r >= offs[0] && r < offs[E]) {
      int lo = 0, hi = E;   // largest e with offs[e] <= r
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offs[mid] <= r) lo = mid; else hi = mid;
      }
      const int64_t i = r - offs[lo];
      const int64_t blk = static_cast<int64_t>(tpre[lo]) + i / bt;
      if (i >= 0 && blk >= 0 && blk < max_blocks) slot = static_cast<int32_t>(blk * 128 + i % bt);
    }
    row_slot[r] = slot;
  }
}

// One thread per (row, 16-block) over ceil(M/128)*128 rows; rows >= M only zero their
// scale-atom bytes. With row_slot (MoE), the threads cover the M rows only and row r's scales go
// to the atom row row_slot[r] (none when it is negative); the caller zeroes the atoms first.
__global__ void act_nvfp4_kernel(const __nv_bfloat16* __restrict__ x, int64_t m, int64_t k,
                                 const float* __restrict__ g_in, const float* __restrict__ partial, int nparts,
                                 const int32_t* __restrict__ row_slot, uint8_t* __restrict__ xq,
                                 uint8_t* __restrict__ xs, float* __restrict__ g_out) {
  __shared__ float red[32];
  __shared__ float g_sh;
  if (g_in == nullptr) {
    float t = 0.f;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) t = fmaxf(t, partial[i]);
    t = warp_max(t);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
      float a = 0.f;
      for (int i = 0; i < static_cast<int>(blockDim.x / 32); ++i) a = fmaxf(a, red[i]);
      g_sh = a > 0.f ? __fdiv_rn(a, 2688.0f) : 1.0f;
    }
  } else if (threadIdx.x == 0) {
    g_sh = *g_in;
  }
  __syncthreads();
  const float g = g_sh;
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  const int64_t blocks_per_row = k / 16;
  const int64_t m_pad = row_slot != nullptr ? m : (m + 127) / 128 * 128;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= m_pad * blocks_per_row) return;
  const int64_t row = i / blocks_per_row, b16 = i % blocks_per_row;
  uint32_t sb = 0;
  if (row < m) {
    const uint4* src = reinterpret_cast<const uint4*>(x + row * k + b16 * 16);
    float f[16];
    float lo8[8], hi8[8];
    bf16x8_to_f32(__ldg(src), lo8);
    bf16x8_to_f32(__ldg(src + 1), hi8);
    float bmax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f[j] = lo8[j];
      f[8 + j] = hi8[j];
      bmax = fmaxf(bmax, fmaxf(fabsf(lo8[j]), fabsf(hi8[j])));
    }
    const uint32_t sbx = e4m3x2(__fdiv_rn(__fdiv_rn(bmax, 6.0f), g), 0.f) & 0xFFu;
    sb = sbx;
    const float denom = __fmul_rn(e4m3_value(sb), g);
    uint32_t bytes[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float a = denom > 0.f ? __fdiv_rn(f[2 * j], denom) : 0.f;
      const float b = denom > 0.f ? __fdiv_rn(f[2 * j + 1], denom) : 0.f;
      bytes[j] = e2m1x2(a, b);
    }
    uint2 out;
    out.x = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
    out.y = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
    *reinterpret_cast<uint2*>(xq + row * (k / 2) + b16 * 8) = out;
  }
  const int64_t arow = row_slot != nullptr ? static_cast<int64_t>(row_slot[row]) : row;
  if (arow < 0) return;
  const int64_t kc = (b16 * 16) / 64;
  const int r = static_cast<int>(arow % 128);
  const int j = static_cast<int>(((b16 * 16) % 64) / 16);
  xs[((arow / 128) * (k / 64) + kc) * kAtomBytes + (r % 32) * 16 + (r / 32) * 4 + j] = static_cast<uint8_t>(sb);
}

__global__ void wait_probe_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    abort_flag = 0u;
  }
  __syncthreads();
  const WaitCtx wc{&abort_flag, err, timeout_ns};
  if (threadIdx.x == 0) {
    (void)mbar_wait(&bar, 0, wc);  // nothing arrives: gives up after timeout_ns
    mbar_arrive(&bar);             // complete the phase so the barrier is left consistent
  }
  __syncthreads();
}

}  // namespace

int act_amax_blocks(int64_t, int64_t) { return kAmaxBlocks; }

__global__ void __launch_bounds__(256) silu_mul_kernel(const __nv_bfloat16* __restrict__ gu,
                                                       __nv_bfloat16* __restrict__ h, int64_t rows,
                                                       int64_t inter) {
  const int64_t per_row = inter / 8;
  const int64_t total = rows * per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row, c8 = i - r * per_row;
    const uint4* row = reinterpret_cast<const uint4*>(gu + r * 2 * inter);
    const uint4 g4 = __ldcs(row + c8);
    const uint4 u4 = __ldcs(row + per_row + c8);
    const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, uw[4] = {u4.x, u4.y, u4.z, u4.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float v[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float g = __uint_as_float(hh ? (gw[q] & 0xFFFF0000u) : (gw[q] << 16));
        const float u = __uint_as_float(hh ? (uw[q] & 0xFFFF0000u) : (uw[q] << 16));
        // logistic(g) from e = exp(-|g|) in (0, 1]: no overflow for very negative gates
        const float e = expf(-fabsf(g));
        v[hh] = g * ((g >= 0.0f ? 1.0f : e) / (1.0f + e)) * u;
      }
      o[q] = pack_bf16x2_rn(v[0], v[1]);
    }
    __stcs(reinterpret_cast<uint4*>(h + r * inter) + c8, make_uint4(o[0], o[1], o[2], o[3]));
  }
}

cudaError_t launch_act_fp8(const __nv_bfloat16* x, int64_t m, int64_t k, uint8_t* xq, float* s_tok,
                           cudaStream_t st) {
  if (m == 0) return cudaSuccess;
  act_fp8_kernel<<<static_cast<unsigned>(m), kFp8Threads, 0, st>>>(x, k, xq, s_tok);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul(const __nv_bfloat16* gu, __nv_bfloat16* h, int64_t rows, int64_t inter, int num_sms,
                            cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int64_t work = rows * (inter / 8);
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;   // 8 blocks of 256 per SM, grid-stride
  if (blocks > cap) blocks = cap;
  silu_mul_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(gu, h, rows, inter);
  return cudaGetLastError();
}

cudaError_t launch_act_nvfp4(const __nv_bfloat16* x, int64_t m, int64_t k, const float* g_in, uint8_t* xq,
                             uint8_t* xs, float* g_out, float* ws, cudaStream_t st) {
  if (m == 0) return cudaSuccess;
  if (g_in == nullptr) amax_bf16_kernel<<<kAmaxBlocks, 256, 0, st>>>(x, m * k / 8, ws);
  const int64_t m_pad = (m + 127) / 128 * 128;
  const int64_t threads = m_pad * (k / 16);
  act_nvfp4_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(x, m, k, g_in, ws, kAmaxBlocks,
                                                                               nullptr, xq, xs, g_out);
  return cudaGetLastError();
}

cudaError_t launch_act_nvfp4_moe(const __nv_bfloat16* x, int64_t rows, int64_t k, const int32_t* offsets, int E,
                                 int bt, int64_t max_blocks, int32_t* row_slot, uint8_t* xq, uint8_t* xs,
                                 float* g_out, float* ws, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  if (E < 1 || E > kSlotMaxExperts) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(xs, 0, static_cast<size_t>(max_blocks) * (k / 64) * kAtomBytes, st);
  if (e != cudaSuccess) return e;
  const int64_t sb = (rows + 1023) / 1024;
  moe_row_slots_kernel<<<static_cast<unsigned>(sb < 1024 ? sb : 1024), 1024, 0, st>>>(offsets, E, rows, bt, max_blocks,
                                                                                      row_slot);
  amax_bf16_kernel<<<kAmaxBlocks, 256, 0, st>>>(x, rows * k / 8, ws);
  const int64_t threads = rows * (k / 16);
  act_nvfp4_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(x, rows, k, nullptr, ws, kAmaxBlocks,
                                                                               row_slot, xq, xs, g_out);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(uint32_t* err, uint64_t timeout_ns, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace hm
