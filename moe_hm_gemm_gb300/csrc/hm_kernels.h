// Kernel parameter blocks and launcher entry points shared between the C ABI (hm_api.cu)
// and the kernel translation units. Internal to libhm.so.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>

#include "hm_sched.cuh"

namespace hm {

// W4A16 GEMM (INT4 or MXFP4 weights restored to bf16, kind::f16 MMA), dense or MoE.
struct F16Params {
  CUtensorMap tmap_x;                 // X bf16 [rows][K], box {64, tile_m}, 128-byte swizzle
  CUtensorMap tmap_x2;                // tensor-core decode kernel: box of two k-blocks (else unused)
  const uint8_t* packed;              // dense: packed weight (header first)
  const uint8_t* const* packed_list;  // MoE: device array of E packed weights, or NULL when the
                                      // experts lie at packed + e * expert_stride
  int64_t expert_stride;              // MoE with packed_list == NULL: bytes between experts
  const int32_t* offsets;             // MoE: expert offsets [E+1]
  __nv_bfloat16* y;                   // [rows][N]
  float* partial;                     // stream-K partial tiles [grid][2][tile_m][128]
  uint32_t* counters;                 // stream-K arrival counters [grid][kCounterSlots], by owner CTA
  uint32_t* err;                      // device error word
  int64_t m, n, k;                    // m = rows
  int32_t fmt;
  int32_t num_experts;
  int32_t num_m_tiles;                // dense only
  int32_t num_n_tiles;
  int32_t group_m;                    // dense: token tiles per group of the tile order (<= 1: m-major)
  SchedParams sched;
  uint64_t timeout_ns;
  uint64_t* trace;                    // optional per-CTA timestamps [grid][16] (diagnostics)
  int32_t cluster;                    // decode kernel: CTAs per cluster (each tile's K ranges), 0/1 = none
  int32_t a_tmem1;                    // tcgen05 W4A16 kernel at 256 tokens: restored weights in TMEM
                                      // beside one accumulator (else in shared memory, two accumulators)
  int32_t epi_scratch;                // tcgen05 W4A16 kernel: the launch has the epilogue's transpose
                                      // scratch (set by the launcher)
  int32_t pair;                       // tcgen05 W4A16 kernel, dense, tile_m 128 or 256: clusters of two
                                      // CTAs share each MMA (sched.grid counts pairs; tmap_x box
                                      // {64, tile_m / 2}; N a multiple of 256)
};

// Block-scaled GEMM (W4A8 MXFP4 x FP8 with kind::mxf8f6f4, W4A4 NVFP4 with kind::mxf4nvf4).
struct MxParams {
  CUtensorMap tmap_w;                 // weight codes (MoE: 3-D, the experts as third dimension)
  CUtensorMap tmap_x;                 // activation codes
  const uint8_t* packed;              // packed weight (header; scale atoms after the codes); MoE: expert 0
  const uint8_t* w_atoms;             // first weight scale atom (MoE: of expert 0)
  const int32_t* offsets;             // MoE: expert offsets [E+1] (device)
  int32_t num_experts;                // MoE: E (0 = dense)
  int64_t expert_stride;              // MoE: bytes between consecutive experts' packed weights
  const uint8_t* x_atoms;             // NVFP4 activation scale atoms
  const float* s_tok;                 // W4A8 per-token scales [M]
  const float* x_global;              // W4A4 activation tensor scale (device scalar)
  __nv_bfloat16* y;
  float* partial;
  uint32_t* counters;
  uint32_t* err;
  int64_t m, n, k;
  int32_t fmt;
  int32_t num_m_tiles;
  int32_t num_n_tiles;
  int32_t k_blocks;                   // K_pad / tile_k
  int32_t group_m;                    // dense: token tiles per group of the tile order (<= 1: m-major)
  SchedParams sched;
  uint64_t timeout_ns;
  uint64_t* trace;
};

// Launch a GEMM kernel with programmatic stream serialization (PDL), so that its prologue and
// weight prefetch overlap the tail of the previous kernel in the stream; the kernel itself
// waits (griddepcontrol.wait) before touching anything the previous kernel may produce or use.
// HM_PDL=0 in the environment launches without the attribute.
template <typename Params>
inline cudaError_t launch_pdl(void (*kern)(Params), int grid, int threads, int smem, cudaStream_t st,
                              const Params& p) {
  static const bool enabled = [] {
    const char* e = std::getenv("HM_PDL");
    return !(e && e[0] == '0');
  }();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = enabled ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Launchers (return a cudaError_t of the launch). `tile_m` and `stages` select an instantiation.
cudaError_t launch_f16_gemm(const F16Params& p, int tile_m, bool moe, cudaStream_t st);
// 128-K blocks per W4A16 load stage for a token tile: the X tensor map for that tile is 2-D
// (box {64, tile_m}) when this is 1 and 3-D (box {64, tile_m, 2*group}) otherwise.
constexpr int f16_group_of(int tile_m) { return tile_m <= 32 ? 4 : (tile_m == 64 ? 2 : 1); }
int f16_group(int tile_m);
cudaError_t launch_mx_gemm(const MxParams& p, int tile_m, cudaStream_t st);
// Grouped (MoE) block-scaled GEMM: p.num_experts >= 1, at most kMxMoeMaxExperts.
constexpr int kMxMoeMaxExperts = 256;
cudaError_t launch_mx_moe_gemm(const MxParams& p, int tile_m, cudaStream_t st);
// The block-scaled kernel runs two CTAs per SM (the plan's grid counts CTAs, not SMs).
constexpr int kMxCtasPerSm = 2;
// Load stages of the W4A16 kernel that serves (fmt, tile_m).
int f16_stages(int fmt, int tile_m, bool a_tmem1 = false, bool pair = false);
// Small-token INT4 kernel (tile_m 16 or 32; hm_gemm_f16s.cu), chosen by launch_f16_gemm unless
// HM_F16_SMALL=0 in the environment.
cudaError_t launch_f16s_gemm(const F16Params& p, int tile_m, bool moe, cudaStream_t st);
int f16s_stages(int tile_m);
bool f16s_serves(int fmt, int tile_m);
int mx_stages(int fmt, int tile_m);
// W4A16 kernel for decode-sized M (hm_gemv.cu): the unit formats (INT4, MXFP4, MXINT4, INT4 in
// groups of 32/64, INT8), up to 32 tokens, warp-level bf16 MMA on registers, split over the packed
// units with a fixed-owner hand-off of shared tiles.
// X comes as tmap_x, a 2-D map with box {128, gemv_tokens(M)} and no swizzle.
constexpr int kGemvMaxTokens = 32;
constexpr int kGemvMoeMaxExperts = 256;   // grouped decode kernel: experts it holds offsets for
constexpr int kGemvMoeTokens = 16;        // grouped decode kernel: the most token rows per tile (8 or 16)
cudaError_t launch_gemv(const F16Params& p, cudaStream_t st);
// Grouped (MoE) decode kernel: expert-sorted rows, token tiles of `tokens` (8 or 16) rows per
// expert, the (tile, k-block) space over all experts cut into one range per CTA (p.sched.grid CTAs;
// the tile count comes from the device offsets); shared tiles hand off through p.partial /
// p.counters.
cudaError_t launch_gemv_moe(const F16Params& p, int tokens, cudaStream_t st);
// Tensor-core decode kernel (hm_gemv_tc.cu): INT4 weights (groups of 128), up to 16 tokens (MoE:
// token tiles of 16 rows), the decode kernel's stream-K split (p.sched.grid CTAs); tmap_x is 3-D
// with box {64, 16, 2} (one 128-K block) and tmap_x2 the same with box {64, 16, 4}.
bool tcdec_serves(int32_t fmt);
int tcdec_stages();
cudaError_t launch_tcdec(const F16Params& p, bool moe, cudaStream_t st);
int gemv_tokens(int64_t m);
int gemv_stages(int64_t m, int32_t fmt);

// Weight preprocessing and activation quantization launchers (hm_weights.cu, hm_act.cu).
cudaError_t launch_quantize_weight(int32_t fmt, int32_t has_zero, int64_t n, int64_t k, int64_t group,
                                   const float* w, const uint8_t* zeros_in, uint8_t* q_out,
                                   void* scales_out, float* g_out, float* ws, cudaStream_t st);
cudaError_t launch_transform(int32_t fmt, int32_t has_zero, int64_t n, int64_t k, float gw, int64_t group,
                             int32_t zconv, const uint8_t* q, const void* scales, const uint8_t* zeros,
                             uint8_t* packed, cudaStream_t st);
cudaError_t launch_dequant(int32_t fmt, int32_t has_zero, int64_t n, int64_t k,
                           const uint8_t* packed, __nv_bfloat16* w, cudaStream_t st);
cudaError_t launch_act_fp8(const __nv_bfloat16* x, int64_t m, int64_t k, uint8_t* xq, float* s_tok,
                           cudaStream_t st);
cudaError_t launch_act_nvfp4(const __nv_bfloat16* x, int64_t m, int64_t k, const float* g_in,
                             uint8_t* xq, uint8_t* xs, float* g_out, float* ws, cudaStream_t st);
int act_amax_blocks(int64_t m, int64_t k);
// NVFP4 quantization of expert-sorted rows for the grouped W4A4 GEMM: codes as the dense layout,
// scale atoms per expert token tile of `bt` rows (at most max_blocks blocks of 128 rows, zeroed
// first); row_slot is [rows] int32 scratch; the tensor scale is computed over all rows.
cudaError_t launch_act_nvfp4_moe(const __nv_bfloat16* x, int64_t rows, int64_t k, const int32_t* offsets, int E,
                                 int bt, int64_t max_blocks, int32_t* row_slot, uint8_t* xq, uint8_t* xs,
                                 float* g_out, float* ws, cudaStream_t st);
// MoE expert activation: h[rows][inter] = bf16(SiLU(gate) * up) from gate_up[rows][2*inter].
cudaError_t launch_silu_mul(const __nv_bfloat16* gu, __nv_bfloat16* h, int64_t rows, int64_t inter, int num_sms,
                            cudaStream_t st);
// MoE token gather (xs[r] = x[token_of_row[r]]) and weighted top-k combine (hm_moe.cu).
cudaError_t launch_moe_gather(const __nv_bfloat16* x, const int32_t* token_of_row, __nv_bfloat16* xs,
                              int64_t tokens, int64_t rows, int64_t k, uint32_t* err, int num_sms,
                              cudaStream_t st);
cudaError_t launch_moe_combine(const __nv_bfloat16* y, const int32_t* pos, const float* w, __nv_bfloat16* out,
                               int64_t tokens, int32_t topk, int64_t rows, int64_t n, uint32_t* err, int num_sms,
                               cudaStream_t st);
// Tensor-core throughput probe (hm_peak.cu): kind 0 kind::f16, 1 kind::mxf8f6f4, 2 kind::mxf4nvf4
// (several issuing warps); 3 and 4 kinds 1 and 2 at N = 256 from one issuer; 5 kind::f16 at N = 256
// with A in TMEM from one issuer, 6 the same with A in shared memory; *flops receives the FLOPs the
// launch issues.
cudaError_t launch_mma_peak(int kind, int32_t iters, int num_sms, uint32_t* err, uint64_t timeout_ns,
                            cudaStream_t st, double* flops);
cudaError_t launch_wait_timeout_probe(uint32_t* err, uint64_t timeout_ns, cudaStream_t st);

}  // namespace hm
