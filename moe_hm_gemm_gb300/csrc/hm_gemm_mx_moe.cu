// Grouped (MoE) block-scaled GEMM instantiations (W4A8 and W4A4 over expert-sorted rows, experts
// at a fixed stride); the kernel is in hm_gemm_mx.cuh.
#include "hm_gemm_mx.cuh"

namespace hm {

cudaError_t launch_mx_moe_gemm(const MxParams& p, int tile_m, cudaStream_t st) {
  if (p.num_experts < 1 || p.num_experts > kMxMoeMaxExperts) return cudaErrorInvalidValue;
  return p.fmt == kW4A4Nv ? launch_bt<true, true>(p, tile_m, st) : launch_bt<false, true>(p, tile_m, st);
}

}  // namespace hm
