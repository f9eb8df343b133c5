// W4A16 GEMM on tcgen05 (kernel in hm_gemm_f16.cuh) for MXFP4 (e2m1 codes) weights with an E8M0
// scale per 32 along K: dense and MoE instantiations over every token tile.
#include "hm_gemm_f16.cuh"

namespace hm {

cudaError_t launch_f16_mxfp4(const F16Params& p, int tile_m, bool moe, cudaStream_t st) {
  return moe ? launch_bt<2, true>(p, tile_m, st) : launch_bt<2, false>(p, tile_m, st);
}

}  // namespace hm
