// W4A16 GEMM on tcgen05 (kernel in hm_gemm_f16.cuh) for INT4 weights with a bf16 scale and u4
// zero-point per 32-K chunk (groups of 32 or 64): dense and MoE instantiations over every token tile.
#include "hm_gemm_f16.cuh"

namespace hm {

cudaError_t launch_f16_int4g(const F16Params& p, int tile_m, bool moe, cudaStream_t st) {
  return moe ? launch_bt<6, true>(p, tile_m, st) : launch_bt<6, false>(p, tile_m, st);
}

}  // namespace hm
