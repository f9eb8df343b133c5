// Dense block-scaled GEMM instantiations (W4A8 and W4A4, token tiles 16..128); the kernel is in
// hm_gemm_mx.cuh.
#include "hm_gemm_mx.cuh"

namespace hm {

int mx_stages(int fmt, int tile_m) {
  const bool nv = fmt == kW4A4Nv;
  switch (tile_m) {
    case 16: return nv ? MxShape<16, true>::kSL : MxShape<16, false>::kSL;
    case 32: return nv ? MxShape<32, true>::kSL : MxShape<32, false>::kSL;
    case 64: return nv ? MxShape<64, true>::kSL : MxShape<64, false>::kSL;
    default: return nv ? MxShape<128, true>::kSL : MxShape<128, false>::kSL;
  }
}

cudaError_t launch_mx_gemm(const MxParams& p, int tile_m, cudaStream_t st) {
  return p.fmt == kW4A4Nv ? launch_bt<true, false>(p, tile_m, st) : launch_bt<false, false>(p, tile_m, st);
}

}  // namespace hm
