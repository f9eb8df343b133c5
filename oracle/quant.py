"""Quantizers and dequantizers, fp64 with explicit fp32 steps (test infrastructure).

Each function restates one quantization recipe step by step. The worked example it
follows for INT4 is on the explainer page "vLLM Humming은 4비트를 어떻게 계산하나",
section "4비트 값에는 스케일이라는 해석 규칙이 붙는다": a weight w is stored as
q = round(w/s) with a signed 4-bit range [-8, 7] (out-of-range values are clamped) and
restored as s*q; the same section attaches one 16-bit scale to every 128 weights. The
page leaves the scale rule, the rounding of the restored value and the zero-point
convention open; the readings taken are:

* scale s = bf16(fp32(max|w| over the group) / 7)  (a bf16 scale per group of 128);
* round = round-half-to-even of the fp32 quotient w/s;
* restored weight = bf16(q*s) (one rounding of the exact product);
* zero-point z (unsigned 4-bit): q = clamp(round(w/s) + z, 0, 15), restored (q - z)*s;
* an all-zero group has s = 0 and q = 0 (resp. q = z).

MXFP4 (OCP Microscaling v1.0, FP4 e2m1 elements, one E8M0 scale per 32): the shared
exponent is floor(log2(amax)) - 2 (2 = largest exponent of e2m1), biased by 127 and
clamped to [0, 254]; elements are RNE(w / 2^(e-127)) saturated to +-6. An all-zero
block has scale code 0 and zero elements.

MXINT4 (named in the news pages' format list, section "하나의 라이브러리로 긴 포맷 목록을
포괄", without a definition): read as the MX scheme of OCP Microscaling v1.0 (one E8M0 shared
exponent per 32 along K) with a signed 4-bit integer element, q in [-8, 7], restored q * X with
X = 2^(e-127). The largest power of two inside the element range is 4 = 2^2, so the shared
exponent takes the same rule as MXFP4: e = clamp(floor(log2 amax) - 2 + 127, 0, 254), which
puts amax / X in [4, 8); elements are clamp(RNE(w / X), -8, 7) (the quotient by a power of two
is exact). This equals OCP's fixed-point reading (MXINT8 style: one integer and two fraction
bits, X' = 2^floor(log2 amax), element q/4) with X = X'/4. An all-zero block has e = 0, q = 0.

FP8 per-token activations (the W4A8 path named on the explainer page, section "가중치
형식, 활성값, 백엔드를 한 줄에 적는다", "BF16 -> per-token FP8"): per row amax;
s_tok = fp32(amax/448); inv = fp32(448/amax); xq = e4m3(RNE, satfinite)(fp32(x*inv)).
A zero row gets s_tok = 0 and xq = 0.

NVFP4 (two-level: e4m3 scale per 16 along K and one fp32 tensor scale): the pages only
name the format; the common recipe is taken: g = fp32(amax_tensor / 2688) (2688 =
448*6); per 16-block sb = e4m3(RNE, satfinite)(fp32(fp32(amax_b/6) / g)); element =
e2m1(RNE, satfinite)(fp32(v / fp32(sb*g))). An all-zero tensor takes g = 1; a block whose
sb is 0 has zero elements.

Parity: pinned in tests/test_oracle_quant.py (page worked example, closed forms,
brute-force scalar loops).
"""
import numpy as np

from .formats import (E4M3, E2M1, bf16r, decode_e2m1, decode_e4m3, decode_e8m0, e2m1_rne,
                      e4m3_rne, f32, round_to)

GROUP_INT4 = 128
GROUP_MX = 32
GROUP_NV = 16


def _groups(w, g):
    w = np.asarray(w, dtype=np.float64)
    n, k = w.shape
    assert k % g == 0
    return w.reshape(n, k // g, g)


# ------------------------------------------------------------------ INT4, group 128

def int4_scales(w, group=GROUP_INT4):
    """s = bf16(fp32(max|w_g|) / 7) per group; returned as float64 values (bf16-exact)."""
    amax = np.abs(_groups(f32(w), group)).max(axis=2)
    return bf16r(f32(f32(amax) / 7.0))


def int4_code(w, s, z=None):
    """One INT4 code: clamp(round(fp32(w/s)) [+ z]) with the page's range [-8, 7] (or [0, 15]
    with a zero-point). s = 0 gives round(...) = 0. Element-wise on arrays."""
    w = np.asarray(w, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(f32(w / s))                       # fp32 quotient, then round half to even
    r = np.where(s == 0, 0.0, r)
    if z is None:
        return np.clip(r, -8, 7).astype(np.int64)
    return np.clip(r + np.asarray(z, dtype=np.float64), 0, 15).astype(np.int64)


def int4_restore(q, s, z=None):
    """Exact restored value (q - z) * s before any rounding."""
    v = np.asarray(q, dtype=np.float64)
    if z is not None:
        v = v - np.asarray(z, dtype=np.float64)
    return v * np.asarray(s, dtype=np.float64)


def quant_int4(w, zeros=None, group=GROUP_INT4):
    """Round-to-nearest INT4 with bf16 group scales.

    Returns (q, s): q int64 [N,K] (signed in [-8,7] without zero-points, unsigned in
    [0,15] with them), s float64 [N,K/group].
    """
    w = f32(w)
    s = int4_scales(w, group)
    s_full = np.repeat(s, group, axis=1)
    z_full = None if zeros is None else np.repeat(np.asarray(zeros), group, axis=1)
    return int4_code(w, s_full, z_full), s


def dequant_int4(q, s, zeros=None, group=GROUP_INT4):
    """Restored weight bf16((q - z) * s), float64 [N,K]."""
    s_full = np.repeat(np.asarray(s, dtype=np.float64), group, axis=1)
    z_full = None if zeros is None else np.repeat(np.asarray(zeros), group, axis=1)
    return bf16r(int4_restore(q, s_full, z_full))


# ------------------------------------------------------------------ INT8 (8-bit integer weights)

def quant_int8(w, zeros=None, group=GROUP_INT4):
    """The page's INT4 rule with the 8-bit integer range (the news pages list integer weights up to
    8 bits, section "하나의 라이브러리로 긴 포맷 목록을 포괄"): s = bf16(fp32(max|w_g|) / 127) per
    group, q = clamp(round(fp32(w / s)), -128, 127), or with an unsigned 8-bit zero-point z,
    clamp(round(fp32(w / s)) + z, 0, 255). Returns (q int64 [N,K], s float64 [N,K/group])."""
    w = f32(w)
    amax = np.abs(_groups(w, group)).max(axis=2)
    s = bf16r(f32(f32(amax) / 127.0))
    s_full = np.repeat(s, group, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(f32(w / s_full))
    r = np.where(s_full == 0, 0.0, r)
    if zeros is None:
        return np.clip(r, -128, 127).astype(np.int64), s
    z_full = np.repeat(np.asarray(zeros, dtype=np.float64), group, axis=1)
    return np.clip(r + z_full, 0, 255).astype(np.int64), s


def dequant_int8(q, s, zeros=None, group=GROUP_INT4):
    """Restored weight bf16((q - z) * s), float64 [N,K] (one rounding of the exact product)."""
    s_full = np.repeat(np.asarray(s, dtype=np.float64), group, axis=1)
    v = np.asarray(q, dtype=np.float64)
    if zeros is not None:
        v = v - np.repeat(np.asarray(zeros, dtype=np.float64), group, axis=1)
    return bf16r(v * s_full)


# ------------------------------------------------------------------ zero-point conventions

def gptq_stored_zero(z):
    """The value a GPTQ-style checkpoint stores for the u4 zero-point z: z - 1, kept in four bits
    (so z = 0 is stored as 15). Reading taken for "zero-points from different quantization tools"
    (aihaber.org, section "Mimari"): such tools keep z - 1 and add the 1 back when restoring."""
    return (np.asarray(z, dtype=np.int64) - 1) % 16


def zero_from_gptq(stored):
    """The zero-point z of a GPTQ-style stored value: stored + 1, modulo 16 (inverse of
    gptq_stored_zero for every z in [0, 15])."""
    return (np.asarray(stored, dtype=np.int64) + 1) % 16


# ------------------------------------------------------------------ MXFP4 (e2m1 + E8M0 / 32)

def mx_scale_codes(w, group=GROUP_MX):
    """E8M0 shared-exponent codes per 32-block along K (OCP MX v1.0 rule)."""
    amax = np.abs(_groups(f32(w), group)).max(axis=2)
    _, e = np.frexp(amax)                            # floor(log2 amax) = e - 1 for amax > 0
    code = np.clip((e - 1) - 2 + 127, 0, 254)
    return np.where(amax == 0, 0, code).astype(np.int64)


def quant_mxfp4(w, group=GROUP_MX):
    """Returns (codes uint8 [N,K] e2m1, scale codes int64 [N,K/32] E8M0)."""
    w = f32(w)
    e = mx_scale_codes(w, group)
    scale = np.repeat(decode_e8m0(e), group, axis=1)
    codes = e2m1_rne(w / scale)                      # division by a power of two is exact
    return codes, e


def dequant_mxfp4(codes, e, group=GROUP_MX):
    """e2m1(code) * 2^(e-127), float64 [N,K] (exact in bf16 for these ranges)."""
    return decode_e2m1(codes) * np.repeat(decode_e8m0(e), group, axis=1)


# ------------------------------------------------------------------ MXINT4 (int4 + E8M0 / 32)

def quant_mxint4(w, group=GROUP_MX):
    """Returns (q int64 [N,K] in [-8, 7], scale codes int64 [N,K/32] E8M0)."""
    w = f32(w)
    e = mx_scale_codes(w, group)
    scale = np.repeat(decode_e8m0(e), group, axis=1)
    q = np.clip(np.rint(w / scale), -8, 7)          # exact quotient, round half to even
    return q.astype(np.int64), e


def dequant_mxint4(q, e, group=GROUP_MX):
    """q * 2^(e-127), float64 [N,K] (exact in bf16: q has at most four significant bits)."""
    return np.asarray(q, dtype=np.float64) * np.repeat(decode_e8m0(e), group, axis=1)


# ------------------------------------------------------------------ FP8 per token

def quant_fp8_per_token(x):
    """x: [M,K] values (bf16-exact). Returns (xq uint8 e4m3 codes [M,K], s_tok float64 [M])."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max(axis=1) if x.shape[1] else np.zeros(x.shape[0])
    with np.errstate(divide="ignore"):
        s_tok = np.where(amax > 0, f32(amax / 448.0), 0.0)
        inv = np.where(amax > 0, f32(448.0 / amax), 0.0)
    xq = e4m3_rne(f32(x * inv[:, None]))
    return xq, s_tok


def dequant_fp8_per_token(xq, s_tok):
    return decode_e4m3(xq) * np.asarray(s_tok, dtype=np.float64)[:, None]


# ------------------------------------------------------------------ NVFP4 (e2m1 + e4m3 / 16 + fp32)

def nvfp4_global_scale(v):
    """g = fp32(amax / 2688), or 1 for an all-zero tensor."""
    amax = float(np.abs(f32(v)).max()) if np.asarray(v).size else 0.0
    return float(f32(amax / 2688.0)) if amax > 0 else 1.0


def quant_nvfp4(v, g=None, group=GROUP_NV):
    """Returns (codes uint8 [R,K] e2m1, block scale codes uint8 [R,K/16] e4m3, g float)."""
    v = f32(v)
    if g is None:
        g = nvfp4_global_scale(v)
    amax_b = np.abs(_groups(v, group)).max(axis=2)
    sb_codes = e4m3_rne(f32(f32(amax_b / 6.0) / g))
    sb = decode_e4m3(sb_codes)
    denom = np.repeat(f32(sb * g), group, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(denom > 0, f32(v / denom), 0.0)
    codes = e2m1_rne(ratio)
    return codes, sb_codes, g


def dequant_nvfp4(codes, sb_codes, g, group=GROUP_NV):
    """e2m1 * sb * g, float64."""
    sb = np.repeat(decode_e4m3(sb_codes), group, axis=1)
    return decode_e2m1(codes) * sb * float(g)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("np",)]
_ = (E4M3, E2M1, round_to)
