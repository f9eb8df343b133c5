/*
 * hm.h — C ABI of libhm.so, a GB300 (sm_103a) library for the weight-quantized linear
 * layer Y[M,N] = X[M,K] * dequant(Wq[N,K])^T and its grouped MoE variant.
 *
 * Method: the Humming quantized-inference kernels as described on the explainer page
 * "vLLM Humming은 4비트를 어떻게 계산하나" (portfolio.ywsung.com): weights are put in a
 * common quantized representation, preprocessed once into a device-friendly layout
 * (section "표현을 맞춘 다음 GPU가 읽기 좋은 배치로 바꾼다"), and combined with activations
 * that arrive per call (same section, figure "Humming의 전처리·세 설정·JIT 컴파일·추론
 * 흐름"). The linear layer is X*W^T with W stored [N,K] (section "같은 가중치도 한
 * 토큰과 많은 토큰에서 비용이 다르다"); MoE splits tokens by expert (same section, MoE
 * paragraph). Formats named on the news pages (news.cocoloop.cn, "하나의 라이브러리로 긴
 * 포맷 목록을 포괄"): W4A16, W4A8, W4A4, MXFP4, MXINT4, NVFP4.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, unless stated otherwise.
 *     The library never allocates device memory; sizes come from the *_size queries.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Calls are
 *     stream-ordered and asynchronous: no host synchronisation, no host reads of device data.
 *   - Arguments are validated on the host before any launch; a failed check returns
 *     HM_ERR_INVALID_ARG / HM_ERR_UNSUPPORTED / HM_ERR_WORKSPACE and launches nothing.
 *     A CUDA launch error returns HM_ERR_CUDA. No C++ exception crosses the ABI.
 *   - Device-side failures (a packed-weight header that does not match the call, or a
 *     pipeline wait that exceeded its time limit) set a device error word that
 *     hm_get_device_error() returns and clears; the kernel then stops its work early.
 *   - All matrices are row-major. bf16 is IEEE bfloat16. Output Y is bf16, rounded once
 *     (nearest-even) from an fp32 accumulator.
 *   - Concurrent calls that share a workspace buffer on different streams race.
 */
#ifndef HM_H_
#define HM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum hm_status {
  HM_OK = 0,
  HM_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, bad offsets length */
  HM_ERR_UNSUPPORTED = 2,   /* format/shape combination not implemented, or a problem whose
                               (tile, 128-K block) space has 2^31 or more iterations */
  HM_ERR_WORKSPACE = 3,     /* workspace smaller than hm_workspace_size() */
  HM_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
  HM_ERR_DEVICE = 5         /* device error word was set (see hm_get_device_error) */
} hm_status;

/* Weight formats.
 *  HM_W4A16_INT4  : INT4 codes, one bf16 scale per 128 along K, optional u4 zero-point per
 *                   group; restored weight bf16((q - z) * s) (z = 0, q signed, when no
 *                   zero-point). bf16 activations, kind::f16 tensor-core MMA.
 *  HM_W4A16_MXFP4 : e2m1 codes with an E8M0 scale per 32 along K (OCP MX v1.0); restored
 *                   e2m1 * 2^(e-127); bf16 activations (the MoE "MXFP4 W4A16" path).
 *  HM_W4A8_MXFP4  : same weights; activations FP8 e4m3 with one fp32 scale per token.
 *  HM_W4A4_NVFP4  : e2m1 codes, e4m3 scale per 16 along K and one fp32 tensor scale, for
 *                   both weights and activations.
 *  HM_W4A16_MXINT4: signed 4-bit integer codes q in [-8, 7] with an E8M0 scale per 32 along K
 *                   (the MX scheme with integer elements, named on the news pages' format
 *                   list, section "하나의 라이브러리로 긴 포맷 목록을 포괄"); restored
 *                   q * 2^(e-127), exact in bf16; bf16 activations.
 *  HM_W4A16_INT4_G32: INT4 as HM_W4A16_INT4 but with a bf16 scale (and optional u4 zero-point)
 *                   per group of 32 or 64 along K (desc.group), the small groups other
 *                   quantization tools produce (aihaber.org, section "Mimari": weights from
 *                   different tools are brought into one standard format); restored
 *                   bf16((q - z) * s) with the group's s and z.
 *  HM_W8A16_INT8  : 8-bit integer codes (signed in [-128, 127], or unsigned in [0, 255] with a u8
 *                   zero-point per group), one bf16 scale per 128 along K, bf16 activations: the
 *                   explainer page's INT4 rule with the 8-bit range (s = bf16(max|w|/127)), one of
 *                   the integer widths of the news pages' format list (up to INT8); restored
 *                   bf16((q - z) * s). */
typedef enum hm_format {
  HM_W4A16_INT4 = 1,
  HM_W4A16_MXFP4 = 2,
  HM_W4A8_MXFP4 = 3,
  HM_W4A4_NVFP4 = 4,
  HM_W4A16_MXINT4 = 5,
  HM_W4A16_INT4_G32 = 6,
  HM_W8A16_INT8 = 7
} hm_format;

/* How zero-points are stored in the standard format handed to hm_transform (INT4 formats with
 * has_zero). HM_ZP_INT: the u4 zero-point z itself, restored (q - z) * s (the convention of
 * AWQ-style checkpoints and of this library). HM_ZP_GPTQ: the value (z - 1) mod 16, as GPTQ-style
 * checkpoints store it; the transform restores z = (stored + 1) mod 16. The packed weight always
 * holds z. hm_quantize_weight takes z itself in either case. */
typedef enum hm_zero_convention { HM_ZP_INT = 0, HM_ZP_GPTQ = 1 } hm_zero_convention;

/* Description of one quantized weight matrix W[N,K] in the common ("standard") format.
 *  has_zero       : integer formats (1, 6 and 7) only; 1 = zero-points present (u4; u8 for 7).
 *  tensor_scale   : HM_W4A4_NVFP4 only; the fp32 per-tensor scale gW (ignored otherwise).
 *  group          : K values per scale. HM_W4A16_INT4: 0 (= 128) or any multiple of 128 that
 *                   divides K, or -1 for one scale per row (per channel, = K); these pack into
 *                   the same units as 128 (each unit carries its group's scale). HM_W4A16_INT4_G32:
 *                   0 (= 32), 32 or 64. HM_W8A16_INT8: 0 or 128. Others: 0 or the format's own
 *                   (32 MX, 16 NVFP4).
 *  zero_convention: hm_zero_convention of the zero-points handed to hm_transform.
 * Shape rules: N >= 1; K % 128 == 0 for formats 1-3 and 5-7, K % 64 == 0 for format 4. */
typedef struct hm_weight_desc {
  int32_t fmt;
  int32_t has_zero;
  int64_t N;
  int64_t K;
  float tensor_scale;
  int32_t group;
  int32_t zero_convention;
} hm_weight_desc;

/* ---------------------------------------------------------------- preprocessing (once) */

/* Bytes of the packed weight buffer for `desc` (256-byte header + padded payload), or 0 if
 * the description is invalid. Host-only, no CUDA call. The payload keeps the byte accounting of
 * the explainer page, section "4비트 값에는 스케일이라는 해석 규칙이 붙는다" (128 INT4 values
 * and one 16-bit scale take 66 bytes), plus one byte per 128 values for INT4 zero-points and one
 * scale byte per 32 (MX) or 16 (NVFP4) values, with N padded to 128 and K to the kernel block as
 * the preprocessing step of section "표현을 맞춘 다음 GPU가 읽기 좋은 배치로 바꾼다" pads them. */
size_t hm_packed_size(const hm_weight_desc* desc);

/* Quantize an fp32 weight W[N,K] (device) into the standard format by round-to-nearest
 * (the explainer page's INT4 rule, section "4비트 값에는 스케일이라는 해석 규칙이 붙는다",
 * generalised per format):
 *   HM_W4A16_INT4 : s = bf16(fp32(max|w| over 128)/7); q = clamp(rne(fp32(w/s)) [+z]) into
 *                   [-8,7] (or [0,15] with the zero-points read from `zeros_in`).
 *   MXFP4 formats : E8M0 e = clamp(floor(log2 amax32) - 2 + 127, 0, 254); code = e2m1(w/2^(e-127)).
 *   HM_W4A16_MXINT4 : the same e (an all-zero block: e = 0); q = clamp(rne(w/2^(e-127)), -8, 7).
 *   HM_W4A4_NVFP4 : g = fp32(amax/2688) computed on the device and written to *g_out;
 *                   sb = e4m3(fp32(fp32(amax16/6)/g)); code = e2m1(fp32(w/fp32(sb*g))).
 *   HM_W8A16_INT8 : s = bf16(fp32(max|w| over 128)/127); q = clamp(rne(fp32(w/s)) [+z]) into
 *                   [-128,127] (or [0,255] with zero-points), one byte per code.
 * Outputs (device): q_out packed codes [N][K/2] ([N][K] bytes for INT8; even k in the low nibble; INT4 and MXINT4
 * nibbles are two's complement, INT4 ones unsigned with zero-points); scales_out [N][K/g]
 * (bf16 for the INT4 formats with g = desc.group; one byte per code for MXFP4 and MXINT4 g=32 and
 * NVFP4 g=16); g_out (NVFP4 only, fp32). INT4 zero-points zeros_in are [N][K/g], one u4 per byte.
 * `ws` needs hm_quantize_workspace_size() bytes (NVFP4 amax partials; may be NULL otherwise). */
size_t hm_quantize_workspace_size(const hm_weight_desc* desc);
hm_status hm_quantize_weight(const hm_weight_desc* desc, const float* w, const uint8_t* zeros_in,
                             void* q_out, void* scales_out, float* g_out, void* ws,
                             size_t ws_bytes, void* stream);

/* Pad and relayout the standard-format weight into `packed` (device, hm_packed_size bytes,
 * 256-byte aligned). Inputs (device): q [N][K/2] packed codes as above; scales [N][K/g];
 * zeros [N][K/g] one u4 value per byte in desc.zero_convention (INT4 formats with has_zero, else
 * NULL), g = desc.group (INT4: a group of 128 j fills j consecutive units with its scale).
 * For HM_W4A4_NVFP4 the header records desc->tensor_scale as gW.
 * Layout: a 256-byte header (magic, fmt, N, K, padded N and K, has_zero, tensor scale, payload
 * bytes), then the payload, N padded to 128 and K to 128 (W4A4: 256):
 *  - INT4, MXFP4-W4A16 and MXINT4: 128x128 "units", n-tile major, each one contiguous block:
 *    8192 bytes of codes (code (r, kk) in the little-endian word at (kk/32)*2048 + r*16 +
 *    ((kk%32)/8)*4, bits 4*((kk%8)/2) + 16*(kk%2); signed codes stored as q + 8), then the
 *    per-row scales (INT4: 128 bf16; MXFP4 and MXINT4: 128 x 4 E8M0) and, for INT4 with
 *    zero-points, 64 bytes of u4 zero-points (row r in the low nibble of byte r/2 when r is
 *    even). Units are 8448 / 8512 / 8704 bytes. HM_W4A16_INT4_G32 units: the same codes, then the
 *    bf16 scale of (row r, 32-K chunk c) at 8192 + 8r + 2c and the u4 zero-point of (r, c) at
 *    9216 + 2r + c/2, bit 4 (c % 2) (a group of 64 fills two chunks); 9216 / 9472 bytes.
 *    HM_W8A16_INT8 units: code (r, kk) as a byte at (kk/16)*2048 + r*16 + kk%16 (q + 128 without
 *    zero-points), 128 bf16 scales at 16384, 128 u8 zero-points at 16640; 16640 / 16768 bytes.
 *  - W4A8 / W4A4: codes row-major [N_pad][K_pad/2], then 512-byte scale atoms
 *    [N_pad/128][K_pad/chunk] (chunk = 128 K for E8M0 per 32, 64 K for e4m3 per 16), the scale
 *    of (row r, sub-block j) at byte (r%32)*16 + (r/32)*4 + j of its atom. */
hm_status hm_transform(const hm_weight_desc* desc, const void* q, const void* scales,
                       const void* zeros, void* packed, void* stream);

/* Test hook: restore the packed weight to bf16 W[N,K] (device). Bit-exact definition of the
 * restored values used by the GEMM (bf16((q-z)*s), e2m1*2^(e-127), or, for NVFP4,
 * bf16(e2m1*sb) without the tensor scale, exact): the "restore s*q" step of the explainer page,
 * section "4비트 값에는 스케일이라는 해석 규칙이 붙는다", which the GEMM kernels perform in
 * registers ("read and unpack", section "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다").
 * w_bf16 must be 16-byte aligned, packed 256-byte aligned; HM_ERR_INVALID_ARG otherwise. A header
 * that does not match `desc` sets device error bit 0 and leaves w_bf16 unwritten. */
hm_status hm_dequant(const hm_weight_desc* desc, const void* packed, void* w_bf16, void* stream);

/* ---------------------------------------------------------------- activations (per call) */

/* Per-token FP8 quantization of bf16 X[M,K] (K % 16 == 0): per row amax; s_tok = fp32(amax/448);
 * inv = fp32(448/amax); xq = e4m3 (RNE, satfinite) of fp32(x*inv). A zero row gives s_tok = 0
 * and xq = 0. Outputs: xq [M][K] bytes, s_tok [M] fp32. (The W4A8 activation path of the
 * explainer page, section "가중치 형식, 활성값, 백엔드를 한 줄에 적는다".) */
hm_status hm_quant_act_fp8(const void* x, int64_t M, int64_t K, void* xq, float* s_tok,
                           void* stream);

/* NVFP4 quantization of bf16 X[M,K] (K % 64 == 0). If `g_in` is non-NULL it is a device fp32
 * holding gX; else gX = fp32(amax(X)/2688) (1 for an all-zero X) is computed on the device
 * (needs `ws` of hm_act_workspace_size bytes). gX is written to *g_out (device fp32).
 * Outputs: codes [M][K/2] (even k low nibble); block scales (e4m3) in 512-byte atoms
 * [ceil(M/128)][K/64], byte (m%32)*16 + ((m%128)/32)*4 + (k%64)/16 within an atom;
 * hm_act_scale_size() bytes. */
size_t hm_act_scale_size(int64_t M, int64_t K);
size_t hm_act_workspace_size(int64_t M, int64_t K);
hm_status hm_quant_act_nvfp4(const void* x, int64_t M, int64_t K, const float* g_in, void* xq,
                             void* xs, float* g_out, void* ws, size_t ws_bytes, void* stream);

/* MoE expert activation between the gate-up and down grouped GEMMs:
 * out[r][c] = bf16(SiLU(gate_up[r][c]) * gate_up[r][inter + c]), SiLU(v) = v / (1 + exp(-v))
 * evaluated in fp32 and rounded once to bf16 (round to nearest even). gate_up: device bf16
 * [rows][2*inter] (gate in the first half of each row, up in the second, as a gate-up GEMM with
 * N = 2*inter writes them); out: device bf16 [rows][inter], not overlapping gate_up.
 * inter % 8 == 0; both pointers 16-byte aligned. rows = 0 is a no-op. Caller owns both buffers;
 * nothing is allocated. (The pages run expert MLPs of the DeepSeek models, the MoE paragraph of
 * the explainer page's section "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다", without
 * printing the activation; the gated SiLU of such experts is the reading taken.)
 * Returns HM_ERR_INVALID_ARG for bad sizes, misaligned or overlapping buffers, HM_ERR_CUDA for a
 * launch failure. */
hm_status hm_silu_mul(const void* gate_up, void* out, int64_t rows, int64_t inter, void* stream);

/* MoE token gather before the gate-up grouped GEMM: xs[r][:] = x[token_of_row[r]][:] for
 * r in [0, rows), an exact copy. x: device bf16 [T][K] (one row per token); token_of_row: device
 * int32 [rows] (the token of each expert-sorted row, rows = T * top-k for a full routing); xs:
 * device bf16 [rows][K], not overlapping x. K % 8 == 0; x and xs 16-byte aligned. rows = 0 is a
 * no-op. A token index outside [0, T) sets device error bit 3 and that row of xs is written as
 * zeros. (The MoE paragraph of the explainer page, section "같은 가중치도 한 토큰과 많은 토큰에서
 * 비용이 다르다": each token goes to the experts it is routed to, and each expert multiplies its
 * own rows; the pages do not print the gather, the plain row copy is the reading taken.)
 * Returns HM_ERR_INVALID_ARG for bad sizes or misaligned pointers, HM_ERR_CUDA for a launch
 * failure. Caller owns every buffer; nothing is allocated. */
hm_status hm_moe_gather(const void* x, const int32_t* token_of_row, void* xs, int64_t T, int64_t rows,
                        int64_t K, void* stream);

/* MoE top-k combine after the down grouped GEMM:
 * out[t][c] = bf16( sum over j = 0 .. topk-1 with pos[t][j] >= 0 of w[t][j] * y[pos[t][j]][c] ),
 * summed in fp32 by one fused multiply-add per slot in slot order, then rounded once to bf16
 * (nearest even); a call is deterministic. y: device bf16 [rows][N] (the expert-sorted outputs);
 * pos: device int32 [T][topk] (the sorted row of token t's j-th routing slot, < 0 = empty slot);
 * w: device fp32 [T][topk] routing weights; out: device bf16 [T][N], not overlapping y.
 * N % 8 == 0; y and out 16-byte aligned. T = 0 is a no-op. A pos >= rows sets device error bit 3
 * and that slot is skipped. (Same passage as hm_moe_gather: the tokens' expert outputs are brought
 * back to the token; the weighted sum of the usual top-k layer is the reading taken.)
 * Returns HM_ERR_INVALID_ARG for bad sizes or misaligned pointers, HM_ERR_CUDA for a launch
 * failure. Caller owns every buffer; nothing is allocated. */
hm_status hm_moe_combine(const void* y, const int32_t* pos, const float* w, void* out, int64_t T,
                         int32_t topk, int64_t rows, int64_t N, void* stream);

/* ---------------------------------------------------------------- GEMM */

/* Workspace bytes hm_gemm / hm_moe_gemm need for this problem (split-K partials and tile
 * counters, internal activation quantization). Host-only. `M` is rows for MoE. The split of K
 * across CTAs for decode-sized M has no passage on the pages (they name only the M-dependent
 * choice of tile shape and stages, aihaber.org, section "Mimari", "Tuning Config"); the
 * workspace holds its fp32 partial tiles. Returns 0 for an invalid format or shape. */
size_t hm_workspace_size(int32_t fmt, int64_t M, int64_t N, int64_t K);

/* The workspace must be zero-filled once after allocation (cudaMemset); the library leaves
 * the counters it uses back at zero after every call, so it can be reused across calls. The
 * counters sit in one fixed block at the start of every workspace (per CTA that owns a tile split
 * along K), which no call writes anything else into: one workspace, sized for the largest of them,
 * may serve calls of every entry (hm_gemm, hm_moe_gemm, hm_moe_gemm_strided) and every size, in
 * stream order. A call that stopped on a device error may leave counters raised: zero the
 * workspace again before reusing it. */

/* Y[M,N] (bf16) = X[M,K] * dequant(W)^T: the linear layer of the explainer page, section
 * "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다" (weights W[N,K] read once and reused
 * over the M rows), with the per-call activations of section "표현을 맞춘 다음 GPU가 읽기 좋은
 * 배치로 바꾼다" (layer(inputs) after transform()) and the A16 / A8 / A4 activation formats of
 * section "가중치 형식, 활성값, 백엔드를 한 줄에 적는다" and the news pages' format list.
 *  HM_W4A16_INT4 / HM_W4A16_MXFP4 / HM_W4A16_MXINT4 : x = bf16 [M][K]; x_scale, x_global ignored.
 *  HM_W4A8_MXFP4 : x = e4m3 [M][K] with x_scale = s_tok fp32 [M]; or, when x_scale is NULL,
 *                  x = bf16 [M][K] quantized internally (hm_quant_act_fp8) into `ws`.
 *                  Y = s_tok[m] * sum_k e4m3(x)*what.
 *  HM_W4A4_NVFP4 : x = codes [M][K/2], x_scale = scale atoms, x_global = device fp32 gX; or,
 *                  when x_scale is NULL, x = bf16 [M][K] quantized internally.
 *                  Y = gX*gW*sum(blocks) sbX*sbW*sum e2m1X*e2m1W.
 * M >= 0 (M = 0 is a no-op), N and K must match the packed header (checked on the device).
 * x must be 16-byte aligned, packed 256-byte aligned. ws: hm_workspace_size bytes.
 * Kernel per call (hm_plan reports it): tcgen05 tensor-core kernels, except the W4A16 formats at
 * decode sizes (M <= 16; 17..32 with MXFP4 and MXINT4, or with INT4 where tcgen05 would split
 * tiles along K),
 * which run on warp-level bf16 MMA with fp32 accumulation (or, with HM_DECODE_TC=1, INT4 up to 16
 * tokens on the tensor-core decode kernel). Output tiles split along K are summed in a fixed
 * order, so a call is deterministic. */
hm_status hm_gemm(int32_t fmt, const void* x, const void* x_scale, const float* x_global,
                  const void* packed, void* y, int64_t M, int64_t N, int64_t K, void* ws,
                  size_t ws_bytes, void* stream);

/* Grouped GEMM over expert-sorted rows (the MoE paragraph of the explainer page, section
 * "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다": tokens are split by expert, so each
 * expert multiplies its own number of rows; the grouped kernel of aihaber.org, section
 * "Performans"): for each expert e, rows
 * [expert_offsets[e], expert_offsets[e+1]) of x are multiplied by expert e's weight:
 * y[r,:] = x[r,:] * dequant(W_e)^T. expert_offsets: device int32 [E+1], non-decreasing,
 * offsets[0] = 0, offsets[E] <= rows (read on the device only; rows from offsets[E] on, e.g.
 * padding, belong to no expert and their y rows are not written). Offsets that decrease, are
 * negative, exceed rows or do not start at 0 set device error bit 2 and nothing is stored.
 * packed: device array of E device pointers, each a packed weight of the same (fmt, N, K).
 * Formats HM_W4A16_INT4 (every group size), HM_W4A16_MXFP4, HM_W4A16_MXINT4 and HM_W8A16_INT8
 * (HM_ERR_UNSUPPORTED otherwise: the block-scaled formats take their experts at a fixed stride,
 * hm_moe_gemm_strided). Experts with no rows cost nothing.
 * ws: hm_moe_workspace_size(fmt, rows, E, N, K) bytes, 16-byte aligned, zero-filled once after
 * allocation (the library leaves it at zero after every call). With E <= 256 and at most 2 rows per
 * expert on average (decode-sized batches) the call runs the grouped decode kernel: warp-level bf16
 * MMA over every expert's (16-row token tile, weight tile, 128-K block) units cut into one range per
 * SM, output tiles split along K summed in a fixed order through ws (deterministic). Otherwise, or
 * when ws is NULL or smaller, the grouped tcgen05 kernel runs (it needs no workspace). */
hm_status hm_moe_gemm(int32_t fmt, const void* x, const int32_t* expert_offsets, int32_t E,
                      const void* const* packed, void* y, int64_t rows, int64_t N, int64_t K,
                      void* ws, size_t ws_bytes, void* stream);

/* Grouped GEMM over expert-sorted rows with the E experts' packed weights back to back in one
 * buffer: expert e's packed weight (header first, as hm_transform writes it) starts at
 * packed + e * expert_stride. Every format, including the block-scaled ones, which need one tensor
 * map over all experts (the explainer page's MoE paragraph, section "같은 가중치도 한 토큰과 많은
 * 토큰에서 비용이 다르다"; the W4A8 MoE of section "가중치 형식, 활성값, 백엔드를 한 줄에 적는다";
 * the grouped NVFP4 path of aihaber.org, section "Performans").
 *  packed: device, 256-byte aligned; expert_stride: a multiple of 256 and at least hm_packed_size()
 *          of one expert's description; every expert's header must match (fmt, N, K), else device
 *          error bit 0 and nothing is stored.
 *  x, x_scale: HM_W4A16_*: x = bf16 [rows][K], x_scale = NULL.
 *          HM_W4A8_MXFP4: x = e4m3 [rows][K] with x_scale = s_tok fp32 [rows]; or x = bf16 and
 *          x_scale = NULL (quantized per token inside the call, into ws).
 *          HM_W4A4_NVFP4: x = bf16 [rows][K], x_scale = NULL; quantized inside the call with one
 *          tensor scale gX = fp32(amax(x)/2688) over all rows and e4m3 scales per 16, the scale atoms
 *          laid out per expert token tile; Y = gX * gW_e * sum ... with gW_e from expert e's header.
 *  expert_offsets, rows, y: as hm_moe_gemm. E <= 1024 (W4A16), <= 256 (W4A8, W4A4).
 *  ws: hm_moe_workspace_size(fmt, rows, E, N, K) bytes. W4A16 formats: as hm_moe_gemm (the grouped
 *      decode kernel's partials and counters; zero-filled once after allocation; NULL runs the
 *      tcgen05 kernel). W4A8 and W4A4: the activations quantized inside the call (0 bytes for W4A8
 *      with x_scale given); need not be zeroed.
 * Returns HM_ERR_INVALID_ARG for bad sizes, strides or pointers, HM_ERR_UNSUPPORTED for W4A4 with
 * x_scale or K % 256 != 0, HM_ERR_WORKSPACE, HM_ERR_CUDA. One launch (plus the activation
 * quantization); tiles m-major within each expert; experts with no rows cost nothing. */
size_t hm_moe_workspace_size(int32_t fmt, int64_t rows, int32_t E, int64_t N, int64_t K);
hm_status hm_moe_gemm_strided(int32_t fmt, const void* x, const void* x_scale, const int32_t* expert_offsets,
                              int32_t E, const void* packed, int64_t expert_stride, void* y, int64_t rows,
                              int64_t N, int64_t K, void* ws, size_t ws_bytes, void* stream);

/* Allocation-free variant of hm_gemm for the W4A16 formats (HM_W4A16_INT4, HM_W4A16_MXFP4,
 * HM_W4A16_MXINT4).
 * The paper has no counterpart; this entry point exists for callers that cannot allocate
 * device memory at all: for example code running inside another engine's fixed memory plan
 * (a plugin that is handed no workspace), or code that must not call cudaMalloc because it
 * synchronises the device. It runs the same kernel as hm_gemm, but the split-K partials and
 * tile counters live in a 20 MiB array inside the library (held by every GPU that loads the
 * library until the process exits), so the caller passes only X, the packed weight and Y.
 * Arguments and layouts are those of hm_gemm. The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine). A plan that shares output tiles between CTAs clears
 * its counters with cudaMemsetAsync on `stream` at every call; a plan in which every CTA owns
 * whole tiles (no stream-K, or stream-K ranges that are whole tiles) uses no scratch at all.
 * Limits: a split plan whose partials (CTAs x 2 x token tile x 128 fp32) and counters exceed
 * 20 MiB returns HM_ERR_WORKSPACE; use hm_gemm with a workspace then. On a 152-SM GB300 the
 * planner's own splits need at most 19 MiB (152 CTAs sharing 128-token tiles), so every M is
 * accepted there; only splits forced through HM_TILE_M / HM_STREAM_K can exceed the array.
 * All calls share the one array: calls that overlap on the GPU (on different streams, or from
 * several threads) race and must be serialised by the caller.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture. */
hm_status hm_gemm_w4a16_noalloc(int32_t fmt, const void* x, const void* packed, void* y,
                                int64_t M, int64_t N, int64_t K, void* stream);

/* ---------------------------------------------------------------- plan / diagnostics */

/* The kernel configuration hm_gemm would use: kernel, token tile, pipeline stages, split
 * (whether CTAs share one output tile along K) and grid size, for a device with `num_sms` SMs.
 * Host-only, no CUDA call. With HM_LOG=1 in the environment, hm_plan, hm_gemm,
 * hm_gemm_w4a16_noalloc and hm_moe_gemm print the configuration they take as one "[hm] ..." line
 * on stderr. */
typedef struct hm_plan_info {
  int32_t bucket;      /* M bucket index: 0: M<=16, 1: <=64, 2: <=256, 3: <=1024, 4: >1024 */
  int32_t tile_m;      /* tokens per tile (tcgen05 MMA N dimension); decode kernel: tokens it
                          is instantiated for (8, 16 or 32, >= M) */
  int32_t tile_n;      /* weight rows per tile (tcgen05 MMA M dimension: 128; 256 when clusters of
                          two CTAs share each MMA, taken only with HM_PAIR=1 in the environment) */
  int32_t tile_k;      /* K per pipeline stage */
  int32_t stages;      /* load-pipeline depth */
  int32_t stream_k;    /* 1 if the K loop is split across CTAs (stream-K) */
  int32_t grid;        /* CTAs launched */
  int32_t tiles;       /* output tiles */
  int32_t kernel;      /* 0: tcgen05 tensor-core kernel; 1: decode kernel (W4A16 formats; warp-level
                          bf16 MMA with fp32 accumulation in registers) for M <= 16, and for
                          17 <= M <= 32 with MXFP4 / MXINT4 or where tcgen05 would split tiles
                          along K; 2: tensor-core decode kernel (INT4, M <= 16, restored weights
                          in TMEM), taken only with HM_DECODE_TC=1 in the environment */
  int32_t sk_tiles;    /* tiles whose K loops are cut into stream-K ranges: 0 without stream-K,
                          else all tiles, or (W4A16 formats with more tiles than CTAs, K loops of
                          64+ blocks, the remainder of tiles over grid at most half a wave) that
                          remainder, run as stream-K ranges over every CTA before the others run
                          whole in full waves; HM_SK_HYBRID=0 / 1 in the environment never / always
                          (remainder up to 90 % of a wave) takes the latter */
} hm_plan_info;
hm_status hm_plan(int32_t fmt, int64_t M, int64_t N, int64_t K, int32_t num_sms,
                  hm_plan_info* out);

/* Returns and clears the device error word on the current device (synchronises `stream`).
 * 0 = no error; bit 0: packed header mismatch; bit 1: pipeline wait timed out;
 * bit 2: bad expert offsets; bit 3: a token or row index of hm_moe_gather / hm_moe_combine out of
 * range. */
uint32_t hm_get_device_error(void* stream);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on an mbarrier
 * nothing will complete, with a limit of `timeout_ns` nanoseconds; the kernel gives up,
 * sets bit 1 of the device error word and returns. */
hm_status hm_debug_wait_timeout(uint64_t timeout_ns, void* stream);

/* Diagnostics: tensor-core throughput probe. Launches one CTA per SM that issues `iters` rounds
 * of MMAs of one tcgen05 kind from shared-memory operands into TMEM accumulators (no memory
 * traffic in the loop): kind 0 = kind::f16 (bf16, M=128, N=256, K=16), 1 = kind::mxf8f6f4
 * block-scaled 1X (e4m3 x e4m3, UE8M0 scales, M=N=128, K=32), 2 = kind::mxf4nvf4 block-scaled 4X
 * (e2m1 x e2m1, UE4M3 scales, M=N=128, K=64), several issuing warps each; kinds 3 and 4 = kinds 1
 * and 2 with N=256 and one issuing warp; kind 5 = kind::f16 with M=128, N=256, K=16, A read from
 * TMEM and one issuing warp (what one issuing thread sustains with the W4A16 kernel's widest
 * instruction); kind 6 = the same with A in shared memory. *flops_out receives the
 * FLOPs (2*M*N*K per MMA) the launch issues; the caller times it on `stream` (events) to get the
 * dense peak of that kind on this device. iters in [1, 2^24]. A completion wait that runs out (2 s)
 * sets device error bit 1. Allocates nothing; the launch holds all of TMEM on each SM. kind in [0, 6]. */
hm_status hm_mma_peak_probe(int32_t kind, int32_t iters, double* flops_out, void* stream);

/* Diagnostics: install (or, with NULL/0, remove) a device buffer of `bytes` bytes on the current
 * device. While installed, each dense W4A16 GEMM launch (grid <= 256 CTAs) writes
 * global-timer stamps of its pipeline milestones per CTA: 0 entry, 1 set-up done, 2 first load
 * issued, 3 last load issued, 4 first weight stage seen by the dequant warps, 6 first MMA,
 * 7 last MMA commit, 8 first accumulator seen by the epilogue, 9 last tile stored, 10 stream-K
 * arrival counted, 11 fix-up done, 12 exit; slot 13 holds the SM id. The buffer must hold
 * 256*16 + 8*64 uint64: after the 256 per-CTA rows, CTA 0 stamps its first 64 load stages and
 * 128-K blocks in eight rows of 64 (row 0: load issued, or in the small-token kernel the block's
 * accumulator seen by the epilogue; dequant start, dequant done; then per block on its MMA
 * issuer: A ready seen, fence passed, MMAs issued, commit issued; last row: the accumulator slot
 * seen free (small-token kernel) or the stage's activation tile seen). The
 * buffer stays owned by the caller; concurrent launches overwrite each other's stamps. */
hm_status hm_set_trace_buffer(void* trace, size_t bytes);

const char* hm_status_string(hm_status s);
const char* hm_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HM_H_ */
