// W4A16 GEMM on tcgen05 (kernel in hm_gemm_f16.cuh): the INT4 instantiations, the stage counts
// the planner reads, and the dispatch over the W4A16 weight formats.
#include <cstdlib>

#include "hm_gemm_f16.cuh"

namespace hm {

int f16_group(int tile_m) { return f16_group_of(tile_m); }

bool f16s_serves(int fmt, int tile_m) {
  if (fmt != kW4A16Int4 || (tile_m != 16 && tile_m != 32)) return false;
  const char* e = std::getenv("HM_F16_SMALL");
  return !(e && e[0] == '0');
}

int f16_stages(int fmt, int tile_m, bool a_tmem1, bool pair) {
  if (pair && (tile_m == 128 || tile_m == 256)) {
    const bool g32 = fmt == kW4A16Int4G, i8 = fmt == kW8A16Int8;
    if (tile_m == 128)
      return i8 ? F16Shape<128, kUnitInt8Zp, false, true>::kSL
                : (g32 ? F16Shape<128, kUnitG32Zp, false, true>::kSL : F16Shape<128, kUnitMx, false, true>::kSL);
    return g32 ? F16Shape<256, kUnitG32Zp, false, true>::kSL : F16Shape<256, kUnitMx, false, true>::kSL;
  }
  if (tile_m == 256 && a_tmem1 && fmt != kW8A16Int8)
    return fmt == kW4A16Int4G ? F16Shape<256, kUnitG32Zp, true>::kSL : F16Shape<256, kUnitMx, true>::kSL;
  if (f16s_serves(fmt, tile_m)) return f16s_stages(tile_m);
  if (fmt == kW8A16Int8) {
    switch (tile_m) {
      case 16: return F16Shape<16, kUnitInt8Zp>::kSL;
      case 32: return F16Shape<32, kUnitInt8Zp>::kSL;
      case 64: return F16Shape<64, kUnitInt8Zp>::kSL;
      case 128: return F16Shape<128, kUnitInt8Zp>::kSL;
      default: return F16Shape<192, kUnitInt8Zp>::kSL;
    }
  }
  if (fmt == kW4A16Int4G) {
    switch (tile_m) {
      case 16: return F16Shape<16, kUnitG32Zp>::kSL;
      case 32: return F16Shape<32, kUnitG32Zp>::kSL;
      case 64: return F16Shape<64, kUnitG32Zp>::kSL;
      case 128: return F16Shape<128, kUnitG32Zp>::kSL;
      case 192: return F16Shape<192, kUnitG32Zp>::kSL;
      default: return F16Shape<256, kUnitG32Zp>::kSL;
    }
  }
  switch (tile_m) {
    case 16: return F16Shape<16>::kSL;
    case 32: return F16Shape<32>::kSL;
    case 64: return F16Shape<64>::kSL;
    case 128: return F16Shape<128>::kSL;
    case 192: return F16Shape<192>::kSL;
    default: return F16Shape<256>::kSL;
  }
}

cudaError_t launch_f16_gemm(const F16Params& p, int tile_m, bool moe, cudaStream_t st) {
  if (f16s_serves(p.fmt, tile_m)) return launch_f16s_gemm(p, tile_m, moe, st);
  if (p.fmt == kW4A16Mx) return launch_f16_mxfp4(p, tile_m, moe, st);
  if (p.fmt == kW4A16MxInt) return launch_f16_mxint4(p, tile_m, moe, st);
  if (p.fmt == kW4A16Int4G) return launch_f16_int4g(p, tile_m, moe, st);
  if (p.fmt == kW8A16Int8) return launch_f16_int8(p, tile_m, moe, st);
  return moe ? launch_bt<0, true>(p, tile_m, st) : launch_bt<0, false>(p, tile_m, st);
}

}  // namespace hm
