// W8A16 GEMM on tcgen05 (kernel in hm_gemm_f16.cuh) for INT8 weights with a bf16 scale (and u8
// zero-point) per 128 along K: dense and MoE instantiations over the token tiles 16..192.
#include "hm_gemm_f16.cuh"

namespace hm {

cudaError_t launch_f16_int8(const F16Params& p, int tile_m, bool moe, cudaStream_t st) {
  return moe ? launch_bt<8, true>(p, tile_m, st) : launch_bt<8, false>(p, tile_m, st);
}

}  // namespace hm
