// Packed-weight and activation layout constants shared by the host API and the kernels.
//
// The preprocessed weight is a 256-byte header followed by a payload (see include/hm.h).
// W4A16 formats are stored as 128x128 "units" (128 weight rows x 128 K), n-tile major, each
// holding the 8 KB of 4-bit codes in the order the dequant warps read them plus the per-row
// scales (and zero-points) of that K block, so one bulk copy fetches everything a pipeline
// stage needs. Inside a unit the code of (row r, column kk) sits in the little-endian 32-bit
// word at byte (kk/32)*2048 + r*16 + ((kk%32)/8)*4, bit 4*((kk%8)/2) + 16*(kk%2): even
// columns fill the low half-word and odd columns the high one, so a mask of 0x000F000F
// after a shift yields a bf16x2 pair of consecutive columns. INT4 nibbles are stored offset
// by 8 when there is no zero-point (u = q + 8), so every INT4 unit restores (u - z) * s. MXINT4
// units hold the same biased nibbles (u = q + 8) with the 128 x 4 E8M0 scales of MXFP4 units.
// INT4 units with a bf16 scale per 32-K chunk (groups of 32 or 64) hold the INT4 nibbles, then the
// scale of (row r, chunk c) at byte 8192 + 8r + 2c and, with zero-points, the u4 zero-point of
// (r, c) at byte 9216 + 2r + c/2, bit 4 (c % 2). INT8 units hold one byte per code, code (r, kk) at
// (kk/16)*2048 + r*16 + kk%16 (q + 128 without zero-points), then 128 bf16 scales at 16384 and,
// with zero-points, 128 u8 zero-points at 16640.
#pragma once
#include <cstdint>

namespace hm {

constexpr uint32_t kMagic = 0x31574D48u;  // "HMW1"
constexpr uint32_t kHeaderBytes = 256;
constexpr int kTileN = 128;               // weight rows per tile (tcgen05 MMA M)
constexpr int kUnitK = 128;               // K per unit / per W4A16 pipeline stage
constexpr uint32_t kUnitCodes = 8192;     // 128 x 128 nibbles
constexpr uint32_t kUnitInt4 = 8448;      // + 128 bf16 scales
constexpr uint32_t kUnitInt4Zp = 8512;    // + 64 bytes of u4 zero-points
constexpr uint32_t kUnitMx = 8704;        // + 128 x 4 E8M0 scales
constexpr uint32_t kUnitG32 = 9216;       // INT4 with a bf16 scale per 32-K chunk: + 128 x 4 bf16
constexpr uint32_t kUnitG32Zp = 9472;     // + 128 x 4 u4 zero-points
constexpr uint32_t kUnitInt8Codes = 16384; // INT8: 128 x 128 bytes of codes
constexpr uint32_t kUnitInt8 = 16640;     // + 128 bf16 scales
constexpr uint32_t kUnitInt8Zp = 16768;   // + 128 u8 zero-points
constexpr uint32_t kAtomBytes = 512;      // scale-factor atom (128 rows x 4 scales)

struct PackedHeader {
  uint32_t magic;
  uint32_t fmt;
  int64_t n;
  int64_t k;
  int64_t n_pad;
  int64_t k_pad;
  uint32_t has_zero;
  float tensor_scale;
  uint64_t payload_bytes;
};
static_assert(sizeof(PackedHeader) == 56, "header layout");

enum Fmt : int32_t {
  kW4A16Int4 = 1, kW4A16Mx = 2, kW4A8Mx = 3, kW4A4Nv = 4, kW4A16MxInt = 5, kW4A16Int4G = 6, kW8A16Int8 = 7
};

// Formats stored as 128x128 units and multiplied with bf16 activations on kind::f16.
__host__ __device__ inline bool unit_fmt(int32_t fmt) {
  return fmt == kW4A16Int4 || fmt == kW4A16Mx || fmt == kW4A16MxInt || fmt == kW4A16Int4G || fmt == kW8A16Int8;
}
// Unit formats whose scales are E8M0 per 32 along K (128 rows x 4 bytes after the codes).
__host__ __device__ inline bool e8_unit_fmt(int32_t fmt) { return fmt == kW4A16Mx || fmt == kW4A16MxInt; }
// Unit formats with a scale per 32-K chunk (E8M0 or, for INT4 in groups of 32 / 64, bf16): no
// small-token kernel, the decode kernel up to 32 tokens.
__host__ __device__ inline bool chunk_scaled_fmt(int32_t fmt) { return e8_unit_fmt(fmt) || fmt == kW4A16Int4G; }

inline int64_t pad_n(int64_t n) { return (n + kTileN - 1) / kTileN * kTileN; }
inline int64_t pad_k(int32_t fmt, int64_t k) { return fmt == kW4A4Nv ? (k + 255) / 256 * 256 : k; }

__host__ __device__ inline uint32_t unit_bytes(int32_t fmt, bool has_zero) {
  if (fmt == kW8A16Int8) return has_zero ? kUnitInt8Zp : kUnitInt8;
  if (fmt == kW4A16Int4G) return has_zero ? kUnitG32Zp : kUnitG32;
  return e8_unit_fmt(fmt) ? kUnitMx : (has_zero ? kUnitInt4Zp : kUnitInt4);
}

inline uint64_t payload_bytes(int32_t fmt, int64_t n, int64_t k, bool has_zero) {
  const int64_t np = pad_n(n), kp = pad_k(fmt, k);
  if (unit_fmt(fmt))
    return static_cast<uint64_t>(np / 128) * (kp / 128) * unit_bytes(fmt, has_zero);
  const int64_t chunk = fmt == kW4A8Mx ? 128 : 64;
  return static_cast<uint64_t>(np) * kp / 2 + static_cast<uint64_t>(np / 128) * (kp / chunk) * kAtomBytes;
}

}  // namespace hm
