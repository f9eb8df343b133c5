// C ABI of libhm.so (declared in include/hm.h): argument validation, the per-M-bucket plan,
// tensor-map encoding, workspace carving and kernel dispatch. Host code only; every step of
// the computation runs in the kernels of the other translation units.
//
// The split between a once-per-layer preprocessing call (hm_transform) and per-call GEMMs
// follows the explainer page "vLLM Humming은 4비트를 어떻게 계산하나", section "표현을 맞춘
// 다음 GPU가 읽기 좋은 배치로 바꾼다" (transform() once, then layer(inputs)); the page's
// "Tuning Config" (tile shape, pipeline stages) is reduced here to a fixed table keyed by
// the M bucket, the device-specific heuristic the news page says Humming also uses
// (news.cocoloop.cn, section "명시된 약점").
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <mutex>

#include "hm.h"
#include "hm_kernels.h"
#include "hm_layout.h"

namespace hm {

__device__ uint32_t g_hm_error;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSmsForSizing = 256;  // workspace queries do not know the device
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per pipeline wait

std::mutex g_mu;
uint32_t* g_err_ptr[kMaxDevices] = {};
uint64_t* g_trace[kMaxDevices] = {};
size_t g_trace_bytes[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

struct DeviceInfo {
  int dev;
  int num_sms;
  uint32_t* err;
};

// Per-device set-up, done once with that device current: SM count and the device address of
// the error word.
bool device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_hm_error) != cudaSuccess) return false;
    g_num_sms[dev] = sms;
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return false;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  out->dev = dev;
  out->num_sms = g_num_sms[dev];
  out->err = g_err_ptr[dev];
  return true;
}

// Trace buffer of the current device if it holds one 16-slot row per CTA of this launch.
uint64_t* trace_for(const DeviceInfo& di, int grid) {
  (void)grid;
  return g_trace_bytes[di.dev] >= static_cast<size_t>(256 * 16 + 8 * 64) * sizeof(uint64_t) ? g_trace[di.dev] : nullptr;
}

uint64_t timeout_ns() {
  const char* s = std::getenv("HM_WAIT_TIMEOUT_NS");
  if (s && *s) return std::strtoull(s, nullptr, 10);
  return kDefaultTimeoutNs;
}

int env_int(const char* name, int dflt) {
  const char* s = std::getenv(name);
  return (s && *s) ? std::atoi(s) : dflt;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_fmt(int32_t f) { return f >= kW4A16Int4 && f <= kW8A16Int8; }

// The K values per scale a description stands for (0 stands for the format's own), or 0 when the
// group, zero-point and convention fields do not fit the format.
int64_t desc_group(const hm_weight_desc* d) {
  const bool int4 = d->fmt == kW4A16Int4 || d->fmt == kW4A16Int4G;
  if (d->has_zero != 0 && d->has_zero != 1) return 0;
  if (d->has_zero && !int4 && d->fmt != kW8A16Int8) return 0;
  if (d->zero_convention != HM_ZP_INT && !(d->zero_convention == HM_ZP_GPTQ && int4 && d->has_zero)) return 0;
  if (d->fmt == kW4A16Int4) {
    const int64_t g = d->group == 0 ? 128 : (d->group == -1 ? d->K : d->group);
    return (g >= 128 && g % 128 == 0 && d->K % g == 0) ? g : 0;
  }
  if (d->fmt == kW4A16Int4G) {
    const int64_t g = d->group == 0 ? 32 : d->group;
    return (g == 32 || g == 64) ? g : 0;
  }
  if (d->fmt == kW8A16Int8) return (d->group == 0 || d->group == 128) ? 128 : 0;
  const int64_t own = d->fmt == kW4A4Nv ? 16 : 32;
  return (d->group == 0 || d->group == own) ? own : 0;
}

bool valid_k(int32_t fmt, int64_t k) {
  if (k <= 0) return false;
  return fmt == kW4A4Nv ? (k % 64 == 0) : (k % 128 == 0);
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Plan {
  int bucket;
  int tile_m;
  int tile_k;
  int stages;
  int stream_k;
  int grid;
  int64_t tiles;
  int64_t num_m_tiles;
  int64_t num_n_tiles;
  int64_t kb_total;
  int gemv;   // 1: a decode kernel (tile_m = tokens it is built for)
  int tc;     // with gemv: the tensor-core decode kernel (else the warp-MMA one)
  int a_tmem1;   // tcgen05 at 256 tokens: restored weights in TMEM beside one accumulator
  int pair;      // tcgen05, dense: clusters of two CTAs share each MMA (tiles of 256 weight rows;
                 // grid counts CTAs, two per pair)
  int64_t sk_tiles;   // with stream_k: the leading tiles in stream-K ranges, the rest whole (0: all)
};

int bucket_of(int64_t m) {
  if (m <= 16) return 0;
  if (m <= 64) return 1;
  if (m <= 256) return 2;
  if (m <= 1024) return 3;
  return 4;
}

// Token tile (tcgen05 MMA N) per M: the smallest of 16/32/64/128 covering M, 128 beyond.
// Token tile (tcgen05 MMA N) per M: the smallest of 16/32/64/128 covering M; beyond 128 the
// W4A16 kernel takes 256 (half the dequant work and X traffic per FLOP) as long as that still
// gives every SM a tile. The block-scaled kernels stop at 128 (TMEM also holds their scale
// factors), and a W4A4 tile narrower than 128 must cover all of M (its activation scale atoms
// hold 128 rows).
// Block-scaled formats above 16 tokens (measured on the W4A8 7168x7168 / 18432x7168 and W4A4
// 8192x8192 layers, M = 32..1024): run tile-parallel with the widest token tile whose tiles fill
// 1.4x the SMs (two CTAs per SM take them); if even 32-token tiles give fewer, run them
// tile-parallel when they still cover 0.9x the SMs, else stream-K. A W4A4 tile narrower than 128
// must cover all of M (its activation scale atoms hold 128 rows), so W4A4 keeps 128, tile-parallel.
struct MxChoice {
  int tile_m;
  bool stream_k;
};
MxChoice mx_choice(int32_t fmt, int64_t m, int64_t n, int num_sms) {
  if (m <= 16) return {16, true};
  if (fmt == kW4A4Nv) return {128, false};
  const int64_t n_tiles = pad_n(n) / 128;
  for (int t : {128, 64, 32})
    if (ceil_div(m, t) * n_tiles * 10 >= static_cast<int64_t>(num_sms) * 14) return {t, false};
  return {32, ceil_div(m, 32) * n_tiles * 10 < static_cast<int64_t>(num_sms) * 9};
}

// INT4 W4A16 for 16 < M <= 512: pick (token tile, stream-K) by a cost model fitted to measured
// times on the 4096x4096, 14336x4096 and 4096x14336 layers at 32..256 rows: time ~ 5 us + blocks
// per CTA x c(tile), where a 128-K block costs c = 0.47 / 0.50 / 0.60 / 0.75 us for tiles of
// 32 / 64 / 128 / 256 tokens, a tile-parallel CTA runs ceil(tiles / SMs) x kb blocks, and a
// stream-K CTA runs ceil(tiles x kb / SMs) blocks plus a hand-off cost of 9 / 16 / 30 / 60
// blocks (the 256-token hand-off, unconstrained by these points, kept at its earlier fit). Narrow
// tiles stream weights faster per block; wide tiles do more tokens per block. With these constants
// the choice is the fastest of the eight (tile, split) configurations at 11 of the 12 measured
// points and within 9 % at the twelfth.
struct F16Choice {
  int tile_m;
  bool stream_k;
};
F16Choice f16_choice(int64_t m, int64_t n, int64_t k, int num_sms) {
  const int64_t n_tiles = pad_n(n) / 128, kb = k / 128;
  const int tiles_m[4] = {32, 64, 128, 256};
  const double cost[4] = {0.47, 0.50, 0.60, 0.75}, handoff[4] = {9, 16, 30, 60};
  F16Choice best{32, true};
  double best_t = 1e30;
  for (int i = 0; i < 4; ++i) {
    const int t = tiles_m[i];
    if (t > 32 && t / 2 >= m) continue;   // no wider than the next power of two covering M
    const int64_t tiles = ceil_div(m, t) * n_tiles;
    const double tp = static_cast<double>(ceil_div(tiles, num_sms) * kb) * cost[i];
    const double sk = (static_cast<double>(ceil_div(tiles * kb, num_sms)) + handoff[i]) * cost[i];
    if (tp < best_t) { best_t = tp; best = {t, false}; }
    if (sk < best_t) { best_t = sk; best = {t, true}; }
  }
  return best;
}

int tile_m_for(int32_t fmt, int64_t m, int64_t n, int num_sms, int64_t k = 0) {
  const bool block_scaled = fmt == kW4A8Mx || fmt == kW4A4Nv;
  const int forced = env_int("HM_TILE_M", 0);
  if (forced == 16 || forced == 32 || forced == 64 || forced == 128 || (forced == 192 && !block_scaled) ||
      (forced == 256 && !block_scaled && fmt != kW8A16Int8)) {
    if (fmt == kW4A4Nv && forced < 128 && m > forced) return 128;
    return forced;
  }
  if (block_scaled) return mx_choice(fmt, m, n, num_sms).tile_m;
  if (fmt == kW4A16Int4 && m > 16 && m <= 512 && k > 0) return f16_choice(m, n, k, num_sms).tile_m;
  if (m <= 16) return 16;
  if (m <= 32) return 32;
  if (m <= 64) return 64;
  if (m <= 128) return 128;
  // The 256-token tile halves the dequant work and X traffic per FLOP; it wins (measured on
  // 4096x4096, 14336x4096, 4096x14336) once its tiles cover about 70 % of the SMs. INT8 units are
  // twice the size: its widest tile is 192 (A in TMEM, three load stages).
  const int64_t n_tiles = pad_n(n) / 128;
  if (fmt == kW8A16Int8) return ceil_div(m, 192) * n_tiles * 10 >= static_cast<int64_t>(num_sms) * 7 ? 192 : 128;
  return ceil_div(m, 256) * n_tiles * 10 >= static_cast<int64_t>(num_sms) * 7 ? 256 : 128;
}

// W4A16 formats at decode-sized M run the warp-MMA decode kernel: with few tokens per weight the
// product is bound by streaming the weights, which the tcgen05 pipeline (restore into TMEM, one
// MMA batch per 128-K block, accumulator hand-offs) does not keep up with (measured on the 4096 and
// 14336 layers). Up to 16 tokens always; for 17..32 tokens MXFP4 and MXINT4 (no small-token
// tcgen05 kernel) always, INT4 when the tcgen05 plan would split tiles along K (the decode
// kernel's K ranges are cheaper there; with a whole tile per CTA the tcgen05 small-token kernel
// is as fast). HM_GEMV=0 keeps tcgen05 for every M; HM_GEMV=2 takes the decode kernel for every M
// it serves (tests, sweeps).
// Decode-sized INT4 layers (up to 16 tokens) may run on the tensor-core decode kernel instead of
// the warp-MMA one (HM_DECODE_TC=1). Off by default: measured on the benchmark layers it is 17-25 %
// slower up to 8 tokens and on par at 16 (a tcgen05.mma of 128 x 16 x 16 costs the issuing SM
// ~40-80 cycles whatever its size, so a 128x128 unit costs ~8 of them as the warp-MMA kernel's 64
// m16n8k16 instructions cost its four sub-partitions).
bool use_tcdec(int32_t fmt, int64_t m) {
  return tcdec_serves(fmt) && m >= 1 && m <= kGemvMoeTokens && env_int("HM_DECODE_TC", 0) == 1;
}

bool use_gemv(int32_t fmt, int64_t m, int64_t n, int64_t k, int num_sms) {
  if (!unit_fmt(fmt)) return false;
  if (m < 1 || m > kGemvMaxTokens) return false;
  const int mode = env_int("HM_GEMV", 1);
  if (mode == 0) return false;
  if (mode == 2 || m <= 16 || fmt != kW4A16Int4) return true;   // no small-token tcgen05 kernel for the others
  return f16_choice(m, n, k, num_sms).stream_k;
}

Plan make_plan(int32_t fmt, int64_t m, int64_t n, int64_t k, int num_sms, bool allow_hybrid = true) {
  Plan p{};
  p.bucket = bucket_of(m);
  if (use_gemv(fmt, m, n, k, num_sms)) {
    p.gemv = 1;
    p.tc = use_tcdec(fmt, m) ? 1 : 0;
    p.tile_m = p.tc ? kGemvMoeTokens : gemv_tokens(m);
    p.tile_k = 128;
    p.stages = p.tc ? tcdec_stages() : gemv_stages(m, fmt);
    p.num_m_tiles = 1;
    p.num_n_tiles = pad_n(n) / 128;
    p.kb_total = k / 128;
    p.tiles = p.num_n_tiles;
    // With no more tiles than SMs, each tile is cut into the same number of K ranges, so every CTA
    // holds one range of one tile: no CTA publishes a shared tile in the middle of its work, and a
    // tile's contributors all finish together. With more tiles than SMs the ranges run across
    // tile boundaries (one range per SM). HM_SK_ALIGN=0 takes the latter everywhere (for sweeps:
    // 112 whole tiles leave 40 of 152 SMs idle).
    if (p.tiles <= num_sms && env_int("HM_SK_ALIGN", 1) != 0) {
      const int64_t per = std::min<int64_t>(num_sms / p.tiles, p.kb_total);
      p.grid = static_cast<int>(p.tiles * per);
    } else {
      p.grid = static_cast<int>(std::min<int64_t>(num_sms, p.tiles * p.kb_total));
    }
    p.stream_k = (p.grid > p.tiles || p.tiles % p.grid != 0) ? 1 : 0;   // some tile shared by CTAs
    return p;
  }
  p.tile_m = tile_m_for(fmt, m, n, num_sms, k);
  p.tile_k = fmt == kW4A4Nv ? 256 : 128;
  p.stages = unit_fmt(fmt) ? f16_stages(fmt, p.tile_m) : mx_stages(fmt, p.tile_m);
  p.num_m_tiles = ceil_div(m > 0 ? m : 1, p.tile_m);
  p.num_n_tiles = pad_n(n) / 128;
  p.kb_total = pad_k(fmt, k) / p.tile_k;
  p.tiles = p.num_m_tiles * p.num_n_tiles;
  // Block-scaled formats run two CTAs per SM, stream-K as mx_choice says. With stream-K over
  // fewer tiles than SMs and tiles wider than 16 tokens, twice the CTAs would split each tile
  // among twice the contributors, and the partials (tile_m x 128 fp32 each) cost more than the
  // second issuer gains: one CTA per SM then.
  const bool block_scaled = fmt == kW4A8Mx || fmt == kW4A4Nv;
  const int sk_env = env_int("HM_STREAM_K", -1);
  // W4A16 with tiles of 128 or 256 tokens: stream-K pays for its partial hand-offs only when a
  // tile's whole K loop is much longer than the balanced share (measured break-even about 30
  // k-blocks); token tiles up to 64 always split.
  const int64_t share = ceil_div(p.tiles * p.kb_total, num_sms);
  const bool modelled = fmt == kW4A16Int4 && m > 16 && m <= 512 && p.tile_m == f16_choice(m, n, k, num_sms).tile_m;
  const bool sk_f16 = modelled ? f16_choice(m, n, k, num_sms).stream_k
                               : p.tiles < num_sms && (p.tile_m <= 64 || p.kb_total > share + 30);
  const bool sk_auto = block_scaled ? (p.tile_m == mx_choice(fmt, m, n, num_sms).tile_m
                                         ? mx_choice(fmt, m, n, num_sms).stream_k
                                         : p.tiles < num_sms)
                                    : sk_f16;
  p.stream_k = sk_env >= 0 ? (sk_env != 0) : (sk_auto ? 1 : 0);
  const int ctas_env = env_int("HM_MX_CTAS_PER_SM", 0);
  const bool one_per_sm = !block_scaled || (ctas_env == 1) ||
                          (ctas_env != 2 && p.stream_k && p.tiles < num_sms && p.tile_m > 16);
  const int64_t ctas = static_cast<int64_t>(num_sms) * (one_per_sm ? 1 : kMxCtasPerSm);
  const int64_t total = p.tiles * p.kb_total;
  const int64_t units = p.stream_k ? total : p.tiles;
  p.grid = static_cast<int>(units < ctas ? units : ctas);
  // Stream-K with no more tiles than CTAs: cut every tile into the same number of K ranges, one
  // per CTA, instead of ranges that run across tile boundaries (HM_SK_ALIGN=0 keeps the latter)
  if (p.stream_k && p.tiles <= ctas && env_int("HM_SK_ALIGN", 1) != 0) {
    const int64_t per = std::min<int64_t>(ctas / p.tiles, p.kb_total);
    p.grid = static_cast<int>(p.tiles * per);
  }
  if (p.grid < 1) p.grid = 1;
  // Hybrid schedule (W4A16 formats, tiles of 128+ tokens, more whole tiles than CTAs): whole waves
  // of tile-parallel work leave the last wave with only tiles mod grid tiles, so those tiles are
  // cut into stream-K ranges over every CTA first and the waves that follow are full. The owner of
  // a shared tile sums the others' fp32 partials (128 KB each at 256 tokens) in 16 dependent
  // chunks, overlapped with its next tile's K loop; measured (256-token tiles, M = 4096 and 8192):
  // +10 % on 4096x14336 at M = 4096 (remainder 37 % of a wave, 112 k-blocks per tile), neutral at a
  // 74 % remainder, and 2-23 % slower on the K = 4096 layers, whose 32-block K loops do not hide
  // the sum. So by default it is taken for K loops of 64+ blocks with a remainder of at most half a
  // wave; HM_SK_HYBRID=1 takes it wherever the remainder fills at most 90 % of a wave and gives
  // every CTA a k-block, HM_SK_HYBRID=0 never; HM_STREAM_K (either value) and HM_PAIR=1 leave it out.
  const int64_t rem = p.tiles % p.grid;
  const int hybrid_env = env_int("HM_SK_HYBRID", -1);
  const bool hybrid_ok = hybrid_env == 1 ? rem * 10 <= static_cast<int64_t>(p.grid) * 9
                                         : hybrid_env != 0 && p.kb_total >= 64 && rem * 2 <= p.grid;
  if (allow_hybrid && unit_fmt(fmt) && !p.stream_k && sk_env < 0 && p.tile_m >= 128 && p.tiles > p.grid &&
      rem > 0 && rem * p.kb_total >= p.grid && hybrid_ok && env_int("HM_PAIR", 0) != 1) {
    p.stream_k = 1;
    p.sk_tiles = rem;
  }
  // 256-token tiles: restored weights in TMEM beside a single accumulator (measured faster on all
  // three benchmark layers from M = 256 on, 9-35 %, once the epilogue stores Y 16 bytes at a time);
  // HM_A_TMEM1=0 keeps them in shared memory with the accumulator pair
  if (p.tile_m == 256 && fmt != kW8A16Int8) {
    p.a_tmem1 = env_int("HM_A_TMEM1", 1) != 0 ? 1 : 0;
    p.stages = f16_stages(fmt, p.tile_m, p.a_tmem1 != 0);
  }
  // CTA pairs (W4A16 formats, whole tiles, 128 or 256 tokens, N a multiple of 256): each pair's
  // tile spans 256 weight rows, and each CTA loads half of the tile's activations.
  const bool pair_ok = unit_fmt(fmt) && !p.stream_k && p.num_n_tiles % 2 == 0 &&
                       (p.tile_m == 128 || (p.tile_m == 256 && fmt != kW8A16Int8)) && num_sms >= 2;
  if (pair_ok && env_int("HM_PAIR", 0) == 1) {
    p.pair = 1;
    p.a_tmem1 = 0;
    p.tiles = p.num_m_tiles * (p.num_n_tiles / 2);
    p.grid = 2 * static_cast<int>(std::min<int64_t>(num_sms / 2, p.tiles));
    p.stages = f16_stages(fmt, p.tile_m, false, true);
  }
  return p;
}

// The kernels walk the (tile, k-block) space in 32-bit indices.
bool plan_fits(const Plan& p) { return p.tiles * p.kb_total < (int64_t{1} << 31); }

// HM_LOG=1: one line on stderr per planned call with the configuration it runs (for sweeps and
// for checking which kernel a layer takes); off by default. Read at every call, so a process may
// switch it on and off.
bool log_on() { return env_int("HM_LOG", 0) != 0; }

void log_plan(const char* entry, int32_t fmt, int64_t m, int64_t n, int64_t k, const Plan& p) {
  if (!log_on()) return;
  std::fprintf(stderr,
               "[hm] %s fmt=%d M=%lld N=%lld K=%lld kernel=%s tile_m=%d tile_k=%d stages=%d stream_k=%d grid=%d "
               "tiles=%lld%s%s",
               entry, fmt, static_cast<long long>(m), static_cast<long long>(n), static_cast<long long>(k),
               p.gemv ? (p.tc ? "decode-tc" : "decode") : "tcgen05", p.tile_m, p.tile_k, p.stages, p.stream_k, p.grid,
               static_cast<long long>(p.tiles), p.a_tmem1 ? " a=tmem" : "", p.pair ? " pair" : "");
  if (p.sk_tiles > 0) std::fprintf(stderr, " sk_tiles=%lld", static_cast<long long>(p.sk_tiles));
  std::fprintf(stderr, "\n");
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WsLayout {
  size_t partial, counters, act_q, act_s, act_g, act_amax, total;
};

// Arrival counters of stream-K tiles, one block per owner CTA ([CTA][kCounterSlots]), at the
// start of every workspace with the same size for every problem and entry: the partials and
// activations of any call start after them, so calls of any size and entry may share a workspace
// (each call leaves the counters at zero).
constexpr size_t kCounterBytes =
    (static_cast<size_t>(kMaxSmsForSizing) * kMxCtasPerSm * kCounterSlots * sizeof(uint32_t) + 255) / 256 * 256;

// The workspace must fit whatever plan any device picks: size the stream-K partials for the
// widest token tile the planner can choose for this M.
WsLayout ws_layout(int32_t fmt, int64_t m, int64_t n, int64_t k, bool internal_act) {
  int widest = tile_m_for(fmt, m, n, 1);          // one SM: the widest choice
  int narrowest = tile_m_for(fmt, m, n, 1 << 30);
  if (fmt == kW4A16Int4 && m > 16 && m <= 512) {  // f16_choice may pick any tile from 32 up to the cover
    narrowest = 32;
    const int cover = m > 128 ? 256 : (m > 64 ? 128 : (m > 32 ? 64 : 32));
    if (cover > widest) widest = cover;
  }
  if (narrowest > widest) widest = narrowest;
  WsLayout w{};
  w.counters = 0;
  size_t off = kCounterBytes;
  w.partial = off;
  const size_t max_ctas = static_cast<size_t>(kMaxSmsForSizing) * ((fmt == kW4A8Mx || fmt == kW4A4Nv) ? kMxCtasPerSm : 1);
  off += align_up(max_ctas * 2 * widest * 128 * sizeof(float));
  w.act_q = w.act_s = w.act_g = w.act_amax = off;
  if (internal_act && fmt == kW4A8Mx) {
    w.act_q = off;
    off += align_up(static_cast<size_t>(m) * k);
    w.act_s = off;
    off += align_up(static_cast<size_t>(m) * sizeof(float));
  } else if (internal_act && fmt == kW4A4Nv) {
    w.act_q = off;
    off += align_up(static_cast<size_t>(m) * k / 2);
    w.act_s = off;
    off += align_up(static_cast<size_t>(ceil_div(m, 128)) * (k / 64) * kAtomBytes);
    w.act_g = off;
    off += align_up(sizeof(float));
    w.act_amax = off;
    off += align_up(static_cast<size_t>(act_amax_blocks(m, k)) * sizeof(float));
  }
  w.total = off;
  return w;
}

hm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? HM_OK : HM_ERR_CUDA; }

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- allocation-free W4A16 GEMM
// Scratch for hm_gemm_w4a16_noalloc: a fixed array in the library's own device memory, so that
// callers who may not allocate still get the split-K schedule. Every GPU that loads the library
// holds these bytes until the process exits.
// 20 MiB: the largest split the planner makes on a 152-SM GB300 (152 CTAs sharing tiles of 128
// tokens) needs 19 MiB of partials plus its counters.
constexpr size_t kNoAllocScratchBytes = size_t(20) << 20;
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
uint8_t* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the array's name is
// only a stand-in for the symbol, never a usable pointer, so the address is looked up once per
// device (with that device current) and cached.
uint8_t* noalloc_scratch(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
  }
  return g_noalloc_ptr[dev];
}

// X (bf16 [rows][K]) as the W4A16 kernel loads it: box {64, tile_m} when a stage holds one
// 128-K block, else the K axis split into 64-element chunks as a third dimension (stride 128
// bytes) so that one load covers the 2*group chunks of a stage.
// CTA pairs load half of a tile's tokens per CTA: box {64, tile_m / 2}.
bool encode_x_f16(CUtensorMap* map, const void* x, int64_t k, int64_t rows, int tile_m, int pair = 0) {
  const int g = f16_group(tile_m);
  if (g == 1) return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, k, rows, k * 2, 64, pair ? tile_m / 2 : tile_m);
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(k / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k * 2), 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(tile_m), static_cast<cuuint32_t>(2 * g)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// X (bf16 [M][K]) as the decode kernel loads it: one box of 128 columns x `tokens` rows per 128-K
// block, unswizzled (rows past M read as zeros).
// Tensor-core decode kernel: X as [K/64 chunks][rows][64], box {64, 16, depth} (depth 2: one
// 128-K block, 4: two), 128-byte swizzle (the MMA's K-major B operand).
bool encode_x_tc(CUtensorMap* map, const void* x, int64_t k, int64_t rows, int depth) {
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(k / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k * 2), 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kGemvMoeTokens), static_cast<cuuint32_t>(depth)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_x_gemv(CUtensorMap* map, const void* x, int64_t k, int64_t m, int tokens) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(m)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k * 2)};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(tokens)};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// X tensor map(s) of a plan's kernel.
bool encode_x_plan(F16Params* prm, const void* x, int64_t k, int64_t m, int gemv, int tc, int tile_m, int pair = 0) {
  if (gemv && tc) return encode_x_tc(&prm->tmap_x, x, k, m, 2) && encode_x_tc(&prm->tmap_x2, x, k, m, 4);
  return gemv ? encode_x_gemv(&prm->tmap_x, x, k, m, tile_m) : encode_x_f16(&prm->tmap_x, x, k, m, tile_m, pair);
}

// Token tile of the grouped GEMM from the mean rows per expert (per-expert counts stay on the
// device); HM_MOE_TILE_M overrides. Block-scaled formats stop at 128. Past 256 rows per expert the
// 256-token tile's halved dequant work per FLOP outweighs its padding of the smaller experts
// (measured: T = 16384, E = 256, top-8 runs 20 % faster than with 128).
int moe_tile_m(int32_t fmt, int64_t rows, int32_t E) {
  const int64_t mean = rows / E;
  int t = mean <= 16 ? 16 : (mean <= 32 ? 32 : (mean <= 64 ? 64 : (mean <= 256 ? 128 : 256)));
  const bool bs = fmt == kW4A8Mx || fmt == kW4A4Nv;
  const int forced = env_int("HM_MOE_TILE_M", 0);
  if (forced == 16 || forced == 32 || forced == 64 || forced == 128 || (forced == 256 && !bs)) t = forced;
  if ((bs || fmt == kW8A16Int8) && t > 128) t = 128;
  return t;
}

// Grouped W4A16 layers with few rows per expert run on the grouped decode kernel: up to 8 rows per
// expert on average it streams the experts' weights faster than the tcgen05 kernel's 16-row tile
// (measured, E = 256 top-8 gate-up and down layers: 1.2-1.3x at T = 16, on par at T = 256).
// HM_MOE_GEMV=0 / 1 forces the choice (given the workspace the decode kernel needs).
bool moe_use_gemv(int32_t fmt, int64_t rows, int32_t E) {
  if (!unit_fmt(fmt) || E > kGemvMoeMaxExperts) return false;
  const int forced = env_int("HM_MOE_GEMV", -1);
  if (forced == 0 || forced == 1) return forced == 1;
  return rows <= 8 * static_cast<int64_t>(E);
}

// Token rows per tile of the grouped decode kernel: 8 halves the MMA work per weight unit, 16 reads
// an expert's weights once for up to 16 rows; HM_MOE_GEMV_TOKENS=8 / 16 forces it.
int moe_gemv_tokens(int64_t rows, int32_t E) {
  const int forced = env_int("HM_MOE_GEMV_TOKENS", 0);
  if (forced == 8 || forced == 16) return forced;
  return rows <= 2 * static_cast<int64_t>(E) ? 8 : 16;
}

// Workspace of the grouped GEMM: the decode kernel's split partials and tile counters (W4A16
// formats), or the block-scaled formats' activations quantized inside the call.
struct MoeWs {
  size_t partial, counters, act_q, act_s, act_g, act_amax, slots, total;
  int64_t max_blocks;
};
MoeWs moe_ws_layout(int32_t fmt, int64_t rows, int32_t E, int64_t n, int64_t k) {
  MoeWs w{};
  w.counters = 0;
  size_t off = kCounterBytes;   // (the counters' place in every workspace)
  (void)n;
  if (unit_fmt(fmt) && E <= kGemvMoeMaxExperts) {
    // the decode kernel's [CTA][token][row] fp32 partials
    w.partial = off;
    off += align_up(static_cast<size_t>(kMaxSmsForSizing) * kGemvMoeTokens * 128 * sizeof(float));
  } else if (fmt == kW4A8Mx) {
    w.act_q = off;
    off += align_up(static_cast<size_t>(rows) * k);
    w.act_s = off;
    off += align_up(static_cast<size_t>(rows) * sizeof(float));
  } else if (fmt == kW4A4Nv) {
    const int bt = moe_tile_m(fmt, rows, E);
    w.max_blocks = ceil_div(rows, bt) + E;
    w.act_q = off;
    off += align_up(static_cast<size_t>(rows) * k / 2);
    w.act_s = off;
    off += align_up(static_cast<size_t>(w.max_blocks) * (k / 64) * kAtomBytes);
    w.act_g = off;
    off += align_up(sizeof(float));
    w.act_amax = off;
    off += align_up(static_cast<size_t>(act_amax_blocks(rows, k)) * sizeof(float));
    w.slots = off;
    off += align_up(static_cast<size_t>(rows) * sizeof(int32_t));
  }
  w.total = off == kCounterBytes ? 0 : off;   // (nothing needed: no workspace)
  return w;
}

// Grouped W4A16 GEMM over expert-sorted rows: the experts' packed weights from a device pointer
// array (list) or at base + e * stride. The grouped decode kernel when moe_use_gemv says so and
// the workspace holds its partials and counters, else the tcgen05 kernel with the token tile of
// moe_tile_m.
hm_status moe_w4a16(int32_t fmt, const void* x, const int32_t* offsets, int32_t E, const uint8_t* const* list,
                    const uint8_t* base, int64_t stride, void* y, int64_t rows, int64_t N, int64_t K, void* ws,
                    size_t ws_bytes, const DeviceInfo& di, cudaStream_t st, const char* entry) {
  // The device-side tile count is at most rows/8 + 1 + E token tiles (of 8 rows or more) per weight tile.
  if ((rows / 8 + 1 + E) * (pad_n(N) / 128) * (K / 128) >= (int64_t{1} << 31)) return HM_ERR_UNSUPPORTED;
  const MoeWs wl = moe_ws_layout(fmt, rows, E, N, K);
  const bool gemv = moe_use_gemv(fmt, rows, E) && ws != nullptr && ws_bytes >= wl.total && aligned(ws, 16) &&
                    di.num_sms <= kMaxSmsForSizing;
  const bool tc = gemv && use_tcdec(fmt, 1);
  const int tile_m = tc ? kGemvMoeTokens : (gemv ? moe_gemv_tokens(rows, E) : moe_tile_m(fmt, rows, E));
  if (log_on())
    std::fprintf(stderr, "[hm] %s fmt=%d E=%d rows=%lld N=%lld K=%lld kernel=%s tile_m=%d grid=%d\n", entry, fmt, E,
                 static_cast<long long>(rows), static_cast<long long>(N), static_cast<long long>(K),
                 gemv ? (tc ? "decode-tc" : "decode") : "tcgen05", tile_m, di.num_sms);
  F16Params prm;
  std::memset(&prm, 0, sizeof(prm));
  if (!encode_x_plan(&prm, x, K, rows, gemv, tc, tile_m)) return HM_ERR_CUDA;
  prm.packed = base;
  prm.packed_list = list;
  prm.expert_stride = stride;
  prm.offsets = offsets;
  prm.y = static_cast<__nv_bfloat16*>(y);
  prm.err = di.err;
  prm.m = rows;
  prm.n = N;
  prm.k = K;
  prm.fmt = fmt;
  prm.num_experts = E;
  prm.num_m_tiles = 0;
  prm.num_n_tiles = static_cast<int32_t>(pad_n(N) / 128);
  prm.sched = SchedParams{0, static_cast<int32_t>(K / 128), di.num_sms, gemv ? 1 : 0};
  prm.timeout_ns = timeout_ns();
  // (256-token tiles: restored weights in TMEM where the epilogue's scratch fits beside the offsets)
  prm.a_tmem1 = tile_m == 256 && fmt != kW8A16Int8 && E <= 512 && env_int("HM_A_TMEM1", 1) != 0 ? 1 : 0;
  if (gemv) {
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    prm.partial = reinterpret_cast<float*>(wsb + wl.partial);
    prm.counters = reinterpret_cast<uint32_t*>(wsb + wl.counters);
    return cuda_status(tc ? launch_tcdec(prm, true, st) : launch_gemv_moe(prm, tile_m, st));
  }
  return cuda_status(launch_f16_gemm(prm, tile_m, true, st));
}

}  // namespace
}  // namespace hm

using namespace hm;

extern "C" {

size_t hm_packed_size(const hm_weight_desc* d) {
  if (d == nullptr || !valid_fmt(d->fmt) || d->N <= 0 || !valid_k(d->fmt, d->K)) return 0;
  if (desc_group(d) == 0) return 0;
  return kHeaderBytes + payload_bytes(d->fmt, d->N, d->K, d->has_zero != 0);
}

size_t hm_quantize_workspace_size(const hm_weight_desc* d) {
  if (d == nullptr || d->fmt != kW4A4Nv) return 0;
  return 512 * sizeof(float);
}

hm_status hm_quantize_weight(const hm_weight_desc* d, const float* w, const uint8_t* zeros_in, void* q_out,
                             void* scales_out, float* g_out, void* ws, size_t ws_bytes, void* stream) {
  if (hm_packed_size(d) == 0 || w == nullptr || q_out == nullptr || scales_out == nullptr)
    return HM_ERR_INVALID_ARG;
  if (d->has_zero && zeros_in == nullptr) return HM_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(q_out, 4)) return HM_ERR_INVALID_ARG;
  if (d->fmt == kW4A4Nv) {
    if (g_out == nullptr) return HM_ERR_INVALID_ARG;
    if (ws == nullptr || ws_bytes < hm_quantize_workspace_size(d)) return HM_ERR_WORKSPACE;
  }
  if (d->fmt != kW4A4Nv && d->K % 128 != 0) return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_quantize_weight(d->fmt, d->has_zero, d->N, d->K, desc_group(d), w, zeros_in,
                                            static_cast<uint8_t*>(q_out), scales_out, g_out,
                                            static_cast<float*>(ws), static_cast<cudaStream_t>(stream)));
}

hm_status hm_transform(const hm_weight_desc* d, const void* q, const void* scales, const void* zeros, void* packed,
                       void* stream) {
  if (hm_packed_size(d) == 0 || q == nullptr || scales == nullptr || packed == nullptr) return HM_ERR_INVALID_ARG;
  if (d->has_zero && zeros == nullptr) return HM_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(q, 16) || !aligned(scales, 4)) return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_transform(d->fmt, d->has_zero, d->N, d->K, d->tensor_scale, desc_group(d),
                                      d->zero_convention,
                                      static_cast<const uint8_t*>(q), scales, static_cast<const uint8_t*>(zeros),
                                      static_cast<uint8_t*>(packed), static_cast<cudaStream_t>(stream)));
}

hm_status hm_dequant(const hm_weight_desc* d, const void* packed, void* w_bf16, void* stream) {
  if (hm_packed_size(d) == 0 || packed == nullptr || w_bf16 == nullptr) return HM_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(w_bf16, 16)) return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_dequant(d->fmt, d->has_zero, d->N, d->K, static_cast<const uint8_t*>(packed),
                                    static_cast<__nv_bfloat16*>(w_bf16), static_cast<cudaStream_t>(stream)));
}

hm_status hm_quant_act_fp8(const void* x, int64_t M, int64_t K, void* xq, float* s_tok, void* stream) {
  if (M < 0 || K <= 0 || K % 16 != 0) return HM_ERR_INVALID_ARG;
  if (M == 0) return HM_OK;
  if (x == nullptr || xq == nullptr || s_tok == nullptr || !aligned(x, 16) || !aligned(xq, 8))
    return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_act_fp8(static_cast<const __nv_bfloat16*>(x), M, K, static_cast<uint8_t*>(xq), s_tok,
                                    static_cast<cudaStream_t>(stream)));
}

hm_status hm_silu_mul(const void* gate_up, void* out, int64_t rows, int64_t inter, void* stream) {
  if (rows < 0 || inter <= 0 || inter % 8 != 0) return HM_ERR_INVALID_ARG;
  if (rows == 0) return HM_OK;
  if (gate_up == nullptr || out == nullptr || !aligned(gate_up, 16) || !aligned(out, 16)) return HM_ERR_INVALID_ARG;
  if (rows > INT64_MAX / (4 * inter)) return HM_ERR_INVALID_ARG;
  // out's rows are half as long as gate_up's, so an overlapping out would overwrite rows not yet read
  const uintptr_t a = reinterpret_cast<uintptr_t>(gate_up), b = reinterpret_cast<uintptr_t>(out);
  if (a < b + static_cast<uintptr_t>(rows * 2 * inter) && b < a + static_cast<uintptr_t>(rows * 4 * inter))
    return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_silu_mul(static_cast<const __nv_bfloat16*>(gate_up), static_cast<__nv_bfloat16*>(out),
                                     rows, inter, di.num_sms, static_cast<cudaStream_t>(stream)));
}

hm_status hm_moe_gather(const void* x, const int32_t* token_of_row, void* xs, int64_t T, int64_t rows, int64_t K,
                        void* stream) {
  if (T < 0 || rows < 0 || K <= 0 || K % 8 != 0) return HM_ERR_INVALID_ARG;
  if (rows == 0) return HM_OK;
  if (x == nullptr || token_of_row == nullptr || xs == nullptr || !aligned(x, 16) || !aligned(xs, 16) ||
      !aligned(token_of_row, 4))
    return HM_ERR_INVALID_ARG;
  if (rows > INT64_MAX / (2 * K)) return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_moe_gather(static_cast<const __nv_bfloat16*>(x), token_of_row,
                                       static_cast<__nv_bfloat16*>(xs), T, rows, K, di.err, di.num_sms,
                                       static_cast<cudaStream_t>(stream)));
}

hm_status hm_moe_combine(const void* y, const int32_t* pos, const float* w, void* out, int64_t T, int32_t topk,
                         int64_t rows, int64_t N, void* stream) {
  if (T < 0 || topk < 1 || rows < 0 || N <= 0 || N % 8 != 0) return HM_ERR_INVALID_ARG;
  if (T == 0) return HM_OK;
  if (y == nullptr || pos == nullptr || w == nullptr || out == nullptr || !aligned(y, 16) || !aligned(out, 16) ||
      !aligned(pos, 4) || !aligned(w, 4))
    return HM_ERR_INVALID_ARG;
  if (T > INT64_MAX / (2 * N) || rows > INT64_MAX / (2 * N)) return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_moe_combine(static_cast<const __nv_bfloat16*>(y), pos, w, static_cast<__nv_bfloat16*>(out),
                                        T, topk, rows, N, di.err, di.num_sms, static_cast<cudaStream_t>(stream)));
}

size_t hm_act_scale_size(int64_t M, int64_t K) {
  if (M < 0 || K <= 0 || K % 64 != 0) return 0;
  return static_cast<size_t>(ceil_div(M, 128)) * (K / 64) * kAtomBytes;
}

size_t hm_act_workspace_size(int64_t M, int64_t K) {
  return static_cast<size_t>(act_amax_blocks(M, K)) * sizeof(float);
}

hm_status hm_quant_act_nvfp4(const void* x, int64_t M, int64_t K, const float* g_in, void* xq, void* xs,
                             float* g_out, void* ws, size_t ws_bytes, void* stream) {
  if (M < 0 || K <= 0 || K % 64 != 0) return HM_ERR_INVALID_ARG;
  if (M == 0) return HM_OK;
  if (x == nullptr || xq == nullptr || xs == nullptr || g_out == nullptr || !aligned(x, 16) || !aligned(xq, 8))
    return HM_ERR_INVALID_ARG;
  if (g_in == nullptr && (ws == nullptr || ws_bytes < hm_act_workspace_size(M, K))) return HM_ERR_WORKSPACE;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_act_nvfp4(static_cast<const __nv_bfloat16*>(x), M, K, g_in, static_cast<uint8_t*>(xq),
                                      static_cast<uint8_t*>(xs), g_out, static_cast<float*>(ws),
                                      static_cast<cudaStream_t>(stream)));
}

size_t hm_workspace_size(int32_t fmt, int64_t M, int64_t N, int64_t K) {
  if (!valid_fmt(fmt) || M < 0 || N <= 0 || !valid_k(fmt, K)) return 0;
  return ws_layout(fmt, M, N, K, true).total;
}

hm_status hm_plan(int32_t fmt, int64_t M, int64_t N, int64_t K, int32_t num_sms, hm_plan_info* out) {
  if (out == nullptr || !valid_fmt(fmt) || M < 0 || N <= 0 || !valid_k(fmt, K) || num_sms <= 0 ||
      num_sms > kMaxSmsForSizing)
    return HM_ERR_INVALID_ARG;
  const Plan p = make_plan(fmt, M, N, K, num_sms);
  log_plan("hm_plan", fmt, M, N, K, p);
  if (!plan_fits(p)) return HM_ERR_UNSUPPORTED;
  out->bucket = p.bucket;
  out->tile_m = p.tile_m;
  out->tile_n = p.pair ? 256 : 128;
  out->tile_k = p.tile_k;
  out->stages = p.stages;
  out->stream_k = p.stream_k;
  out->grid = p.grid;
  out->tiles = static_cast<int32_t>(p.tiles);
  out->kernel = p.gemv ? (p.tc ? 2 : 1) : 0;
  out->sk_tiles = static_cast<int32_t>(p.stream_k ? (p.sk_tiles > 0 ? p.sk_tiles : p.tiles) : 0);
  return HM_OK;
}

hm_status hm_gemm(int32_t fmt, const void* x, const void* x_scale, const float* x_global, const void* packed,
                  void* y, int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes, void* stream) {
  if (!valid_fmt(fmt) || M < 0 || N <= 0 || !valid_k(fmt, K)) return HM_ERR_INVALID_ARG;
  if (M == 0) return HM_OK;
  if (x == nullptr || packed == nullptr || y == nullptr) return HM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(packed, 256) || !aligned(y, 4) || (N % 2) != 0) return HM_ERR_INVALID_ARG;
  if (fmt == kW4A4Nv && K % 256 != 0) return HM_ERR_UNSUPPORTED;  // GEMM K blocks are 256 wide
  const bool internal_act = (fmt == kW4A8Mx || fmt == kW4A4Nv) && x_scale == nullptr;
  if (fmt == kW4A4Nv && !internal_act && x_global == nullptr) return HM_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(fmt, M, N, K, internal_act);
  if (ws == nullptr || ws_bytes < wl.total) return HM_ERR_WORKSPACE;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Plan p = make_plan(fmt, M, N, K, di.num_sms);
  log_plan("hm_gemm", fmt, M, N, K, p);
  if (!plan_fits(p)) return HM_ERR_UNSUPPORTED;
  uint8_t* wsb = static_cast<uint8_t*>(ws);

  if (unit_fmt(fmt)) {
    F16Params prm;
    std::memset(&prm, 0, sizeof(prm));
    if (!encode_x_plan(&prm, x, K, M, p.gemv, p.tc, p.tile_m, p.pair))
      return HM_ERR_CUDA;
    prm.packed = static_cast<const uint8_t*>(packed);
    prm.y = static_cast<__nv_bfloat16*>(y);
    prm.partial = reinterpret_cast<float*>(wsb + wl.partial);
    prm.counters = reinterpret_cast<uint32_t*>(wsb + wl.counters);
    prm.err = di.err;
    prm.m = M;
    prm.n = N;
    prm.k = K;
    prm.fmt = fmt;
    prm.num_experts = 0;
    prm.num_m_tiles = static_cast<int32_t>(p.num_m_tiles);
    prm.num_n_tiles = static_cast<int32_t>(p.num_n_tiles);
    // HM_F16_GROUP=g: grouped tile order (measured neutral, +-3 %, on the W4A16 layers; m-major by default)
    prm.group_m = env_int("HM_F16_GROUP", 0);
    prm.sched = SchedParams{static_cast<int32_t>(p.tiles), static_cast<int32_t>(p.kb_total),
                            p.pair ? p.grid / 2 : p.grid, p.stream_k, static_cast<int32_t>(p.sk_tiles)};
    prm.timeout_ns = timeout_ns();
    prm.a_tmem1 = p.a_tmem1;
    prm.pair = p.pair;
    prm.trace = trace_for(di, p.grid);
    if (p.gemv) return cuda_status(p.tc ? launch_tcdec(prm, false, st) : launch_gemv(prm, st));
    return cuda_status(launch_f16_gemm(prm, p.tile_m, false, st));
  }

  // Block-scaled formats: quantize bf16 activations first when the caller passed none.
  const uint8_t* xq = static_cast<const uint8_t*>(x);
  const void* xs = x_scale;
  const float* xg = x_global;
  if (internal_act) {
    if (!aligned(x, 16)) return HM_ERR_INVALID_ARG;
    uint8_t* q = wsb + wl.act_q;
    if (fmt == kW4A8Mx) {
      float* s = reinterpret_cast<float*>(wsb + wl.act_s);
      const cudaError_t e = launch_act_fp8(static_cast<const __nv_bfloat16*>(x), M, K, q, s, st);
      if (e != cudaSuccess) return HM_ERR_CUDA;
      xs = s;
    } else {
      float* g = reinterpret_cast<float*>(wsb + wl.act_g);
      const cudaError_t e = launch_act_nvfp4(static_cast<const __nv_bfloat16*>(x), M, K, nullptr, q,
                                             wsb + wl.act_s, g, reinterpret_cast<float*>(wsb + wl.act_amax), st);
      if (e != cudaSuccess) return HM_ERR_CUDA;
      xs = wsb + wl.act_s;
      xg = g;
    }
    xq = q;
  }
  MxParams prm;
  std::memset(&prm, 0, sizeof(prm));
  const int64_t n_pad = pad_n(N), k_pad = pad_k(fmt, K);
  const uint8_t* body = static_cast<const uint8_t*>(packed) + kHeaderBytes;
  bool ok;
  if (fmt == kW4A8Mx) {
    // weights: e2m1 codes, expanded by TMA to one byte per code in shared memory
    ok = encode_2d(&prm.tmap_w, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, body, k_pad, n_pad, k_pad / 2, 128, 128) &&
         encode_2d(&prm.tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, K, M, K, 128, p.tile_m);
  } else {
    ok = encode_2d(&prm.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, body, k_pad / 2, n_pad, k_pad / 2, 128, 128) &&
         encode_2d(&prm.tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, K / 2, M, K / 2, 128, p.tile_m);
  }
  if (!ok) return HM_ERR_CUDA;
  prm.packed = static_cast<const uint8_t*>(packed);
  prm.w_atoms = body + static_cast<size_t>(n_pad) * k_pad / 2;
  prm.x_atoms = static_cast<const uint8_t*>(xs);
  prm.s_tok = static_cast<const float*>(xs);
  prm.x_global = xg;
  prm.y = static_cast<__nv_bfloat16*>(y);
  prm.partial = reinterpret_cast<float*>(wsb + wl.partial);
  prm.counters = reinterpret_cast<uint32_t*>(wsb + wl.counters);
  prm.err = di.err;
  prm.m = M;
  prm.n = N;
  prm.k = K;
  prm.fmt = fmt;
  prm.num_m_tiles = static_cast<int32_t>(p.num_m_tiles);
  prm.num_n_tiles = static_cast<int32_t>(p.num_n_tiles);
  prm.k_blocks = static_cast<int32_t>(p.kb_total);
  // grouped tile order, 16 token tiles per group (measured +3-12 % W4A8 and +5-10 % W4A4 at
  // M >= 1024 over the m-major order, whose waves re-read every weight tile from DRAM);
  // HM_MX_GROUP=0 keeps the m-major order
  prm.group_m = env_int("HM_MX_GROUP", 16);
  prm.sched = SchedParams{static_cast<int32_t>(p.tiles), static_cast<int32_t>(p.kb_total), p.grid, p.stream_k};
  prm.timeout_ns = timeout_ns();
  const cudaError_t e = launch_mx_gemm(prm, p.tile_m, st);
  if (e == cudaErrorNotSupported) return HM_ERR_UNSUPPORTED;
  return cuda_status(e);
}

hm_status hm_moe_gemm(int32_t fmt, const void* x, const int32_t* expert_offsets, int32_t E,
                      const void* const* packed, void* y, int64_t rows, int64_t N, int64_t K, void* ws,
                      size_t ws_bytes, void* stream) {
  if (!unit_fmt(fmt)) return valid_fmt(fmt) ? HM_ERR_UNSUPPORTED : HM_ERR_INVALID_ARG;
  if (rows < 0 || N <= 0 || !valid_k(fmt, K) || E < 1 || E > 1024) return HM_ERR_INVALID_ARG;
  if (rows == 0) return HM_OK;
  if (x == nullptr || expert_offsets == nullptr || packed == nullptr || y == nullptr) return HM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 4) || (N % 2) != 0 || !aligned(packed, 8)) return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return moe_w4a16(fmt, x, expert_offsets, E, reinterpret_cast<const uint8_t* const*>(packed), nullptr, 0, y, rows, N,
                   K, ws, ws_bytes, di, cudaStream_t(stream), "hm_moe_gemm");
}

size_t hm_moe_workspace_size(int32_t fmt, int64_t rows, int32_t E, int64_t N, int64_t K) {
  if (!valid_fmt(fmt) || rows < 0 || E < 1 || N <= 0 || !valid_k(fmt, K)) return 0;
  return moe_ws_layout(fmt, rows, E, N, K).total;
}

hm_status hm_moe_gemm_strided(int32_t fmt, const void* x, const void* x_scale, const int32_t* expert_offsets, int32_t E,
                              const void* packed, int64_t expert_stride, void* y, int64_t rows, int64_t N, int64_t K,
                              void* ws, size_t ws_bytes, void* stream) {
  if (!valid_fmt(fmt) || rows < 0 || N <= 0 || !valid_k(fmt, K) || E < 1 || E > 1024) return HM_ERR_INVALID_ARG;
  if (rows == 0) return HM_OK;
  if (x == nullptr || expert_offsets == nullptr || packed == nullptr || y == nullptr) return HM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 4) || (N % 2) != 0 || !aligned(packed, 256) || !aligned(expert_offsets, 4))
    return HM_ERR_INVALID_ARG;
  // (INT4 without zero-points packs smaller; either size may be passed as the stride, and every
  // expert's header is checked on the device)
  hm_weight_desc d0{fmt, 0, N, K, 1.0f, 0, 0};
  if (expert_stride < static_cast<int64_t>(hm_packed_size(&d0)) || expert_stride % 256 != 0) return HM_ERR_INVALID_ARG;
  const bool bs = fmt == kW4A8Mx || fmt == kW4A4Nv;
  if (fmt == kW4A4Nv && (x_scale != nullptr || K % 256 != 0)) return HM_ERR_UNSUPPORTED;
  if (bs && E > kMxMoeMaxExperts) return HM_ERR_UNSUPPORTED;
  const MoeWs wl = moe_ws_layout(fmt, rows, E, N, K);
  if (bs && x_scale == nullptr && (ws == nullptr || ws_bytes < wl.total)) return HM_ERR_WORKSPACE;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!bs)
    return moe_w4a16(fmt, x, expert_offsets, E, nullptr, static_cast<const uint8_t*>(packed), expert_stride, y, rows,
                     N, K, ws, ws_bytes, di, st, "hm_moe_gemm_strided");
  const int tile_m = moe_tile_m(fmt, rows, E);
  if (log_on())
    std::fprintf(stderr, "[hm] hm_moe_gemm_strided fmt=%d E=%d rows=%lld N=%lld K=%lld tile_m=%d\n", fmt, E,
                 static_cast<long long>(rows), static_cast<long long>(N), static_cast<long long>(K), tile_m);
  const int64_t n_pad = pad_n(N), k_pad = pad_k(fmt, K);
  if ((rows / 16 + 1 + E) * (n_pad / 128) * (k_pad / (fmt == kW4A4Nv ? 256 : 128)) >= (int64_t{1} << 31))
    return HM_ERR_UNSUPPORTED;
  const bool internal_act = x_scale == nullptr;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const uint8_t* xq = static_cast<const uint8_t*>(x);
  const void* xs = x_scale;
  const float* xg = nullptr;
  if (internal_act) {
    uint8_t* q = wsb + wl.act_q;
    if (fmt == kW4A8Mx) {
      float* sp = reinterpret_cast<float*>(wsb + wl.act_s);
      if (launch_act_fp8(static_cast<const __nv_bfloat16*>(x), rows, K, q, sp, st) != cudaSuccess) return HM_ERR_CUDA;
      xs = sp;
    } else {
      float* g = reinterpret_cast<float*>(wsb + wl.act_g);
      if (launch_act_nvfp4_moe(static_cast<const __nv_bfloat16*>(x), rows, K, expert_offsets, E, tile_m, wl.max_blocks,
                               reinterpret_cast<int32_t*>(wsb + wl.slots), q, wsb + wl.act_s, g,
                               reinterpret_cast<float*>(wsb + wl.act_amax), st) != cudaSuccess)
        return HM_ERR_CUDA;
      xs = wsb + wl.act_s;
      xg = g;
    }
    xq = q;
  }
  MxParams prm;
  std::memset(&prm, 0, sizeof(prm));
  const uint8_t* body = static_cast<const uint8_t*>(packed) + kHeaderBytes;
  {
    const bool w8 = fmt == kW4A8Mx;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(w8 ? k_pad : k_pad / 2), static_cast<cuuint64_t>(n_pad),
                                static_cast<cuuint64_t>(E)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k_pad / 2), static_cast<cuuint64_t>(expert_stride)};
    const cuuint32_t box[3] = {128, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (g_encode(&prm.tmap_w, w8 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                 const_cast<uint8_t*>(body), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return HM_ERR_CUDA;
    const bool ok = w8 ? encode_2d(&prm.tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, K, rows, K, 128, tile_m)
                       : encode_2d(&prm.tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, K / 2, rows, K / 2, 128, tile_m);
    if (!ok) return HM_ERR_CUDA;
  }
  prm.packed = static_cast<const uint8_t*>(packed);
  prm.w_atoms = body + static_cast<size_t>(n_pad) * k_pad / 2;
  prm.offsets = expert_offsets;
  prm.num_experts = E;
  prm.expert_stride = expert_stride;
  prm.x_atoms = static_cast<const uint8_t*>(xs);
  prm.s_tok = static_cast<const float*>(xs);
  prm.x_global = xg;
  prm.y = static_cast<__nv_bfloat16*>(y);
  prm.err = di.err;
  prm.m = rows;
  prm.n = N;
  prm.k = K;
  prm.fmt = fmt;
  prm.num_m_tiles = 0;
  prm.num_n_tiles = static_cast<int32_t>(n_pad / 128);
  prm.k_blocks = static_cast<int32_t>(k_pad / (fmt == kW4A4Nv ? 256 : 128));
  prm.sched = SchedParams{0, prm.k_blocks, di.num_sms * kMxCtasPerSm, 0};
  prm.timeout_ns = timeout_ns();
  const cudaError_t e = launch_mx_moe_gemm(prm, tile_m, st);
  if (e == cudaErrorNotSupported) return HM_ERR_UNSUPPORTED;
  return cuda_status(e);
}

hm_status hm_gemm_w4a16_noalloc(int32_t fmt, const void* x, const void* packed, void* y, int64_t M, int64_t N,
                                int64_t K, void* stream) {
  if (!unit_fmt(fmt) || M < 0 || N <= 0 || !valid_k(fmt, K)) return HM_ERR_INVALID_ARG;
  if (M == 0) return HM_OK;
  if (x == nullptr || packed == nullptr || y == nullptr) return HM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(packed, 256) || !aligned(y, 4) || (N % 2) != 0) return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  uint8_t* scratch = noalloc_scratch(di.dev);
  if (scratch == nullptr) return HM_ERR_CUDA;
  Plan p = make_plan(fmt, M, N, K, di.num_sms);
  // A hybrid schedule whose stream-K partials do not fit the scratch runs whole waves instead.
  if (p.sk_tiles > 0 && align_up(static_cast<size_t>(p.grid) * 2 * p.tile_m * 128 * sizeof(float)) +
                                align_up(static_cast<size_t>(p.grid) * kCounterSlots * sizeof(uint32_t)) >
                            kNoAllocScratchBytes)
    p = make_plan(fmt, M, N, K, di.num_sms, false);
  log_plan("hm_gemm_w4a16_noalloc", fmt, M, N, K, p);
  if (!plan_fits(p)) return HM_ERR_UNSUPPORTED;
  // The arrival counters of this launch's CTAs, then their partials. Only a plan that shares tiles
  // between CTAs touches them: without stream-K, or with stream-K ranges that cover whole tiles (as
  // many CTAs as tiles, or a whole number of tiles per CTA), every CTA owns its tiles outright and
  // the call needs no scratch at all.
  const bool shared = p.stream_k && (p.grid > p.tiles || p.tiles % p.grid != 0);
  const size_t counter_bytes = shared ? align_up(static_cast<size_t>(p.grid) * kCounterSlots * sizeof(uint32_t)) : 0;
  const size_t partial_bytes =
      shared ? align_up(static_cast<size_t>(p.grid) * 2 * p.tile_m * 128 * sizeof(float)) : 0;
  if (partial_bytes + counter_bytes > kNoAllocScratchBytes) return HM_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The counters must start at zero; clear them on every call (cheap, and safe even after a
  // call that stopped early on a device error).
  if (shared && cudaMemsetAsync(scratch, 0, counter_bytes, st) != cudaSuccess) return HM_ERR_CUDA;
  F16Params prm;
  std::memset(&prm, 0, sizeof(prm));
  if (!encode_x_plan(&prm, x, K, M, p.gemv, p.tc, p.tile_m, p.pair))
    return HM_ERR_CUDA;
  prm.packed = static_cast<const uint8_t*>(packed);
  prm.y = static_cast<__nv_bfloat16*>(y);
  prm.counters = reinterpret_cast<uint32_t*>(scratch);
  prm.partial = reinterpret_cast<float*>(scratch + counter_bytes);
  prm.err = di.err;
  prm.m = M;
  prm.n = N;
  prm.k = K;
  prm.fmt = fmt;
  prm.num_m_tiles = static_cast<int32_t>(p.num_m_tiles);
  prm.num_n_tiles = static_cast<int32_t>(p.num_n_tiles);
  prm.sched = SchedParams{static_cast<int32_t>(p.tiles), static_cast<int32_t>(p.kb_total),
                          p.pair ? p.grid / 2 : p.grid, p.stream_k, static_cast<int32_t>(p.sk_tiles)};
  prm.timeout_ns = timeout_ns();
  prm.a_tmem1 = p.a_tmem1;
  prm.pair = p.pair;
  return cuda_status(p.gemv ? (p.tc ? launch_tcdec(prm, false, st) : launch_gemv(prm, st))
                            : launch_f16_gemm(prm, p.tile_m, false, st));
}

uint32_t hm_get_device_error(void* stream) {
  DeviceInfo di;
  if (!device_info(&di)) return 0xFFFFFFFFu;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_hm_error, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return 0xFFFFFFFFu;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbolAsync(g_hm_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return 0xFFFFFFFFu;
  if (cudaStreamSynchronize(st) != cudaSuccess) return 0xFFFFFFFFu;
  return v;
}

hm_status hm_debug_wait_timeout(uint64_t timeout_ns_, void* stream) {
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_wait_timeout_probe(di.err, timeout_ns_, static_cast<cudaStream_t>(stream)));
}

hm_status hm_mma_peak_probe(int32_t kind, int32_t iters, double* flops_out, void* stream) {
  if (kind < 0 || kind > 6 || iters < 1 || iters > (1 << 24) || flops_out == nullptr) return HM_ERR_INVALID_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  return cuda_status(launch_mma_peak(kind, iters, di.num_sms, di.err, kDefaultTimeoutNs,
                                     static_cast<cudaStream_t>(stream), flops_out));
}

const char* hm_status_string(hm_status s) {
  switch (s) {
    case HM_OK: return "ok";
    case HM_ERR_INVALID_ARG: return "invalid argument";
    case HM_ERR_UNSUPPORTED: return "unsupported format or shape";
    case HM_ERR_WORKSPACE: return "workspace too small";
    case HM_ERR_CUDA: return "CUDA error";
    case HM_ERR_DEVICE: return "device error word set";
  }
  return "unknown status";
}

hm_status hm_set_trace_buffer(void* trace, size_t bytes) {
  DeviceInfo di;
  if (!device_info(&di)) return HM_ERR_CUDA;
  if ((trace == nullptr) != (bytes == 0) || !aligned(trace, 8)) return HM_ERR_INVALID_ARG;
  g_trace[di.dev] = static_cast<uint64_t*>(trace);
  g_trace_bytes[di.dev] = bytes;
  return HM_OK;
}

const char* hm_version(void) { return "hm 0.1.0 (sm_103a)"; }

}  // extern "C"
