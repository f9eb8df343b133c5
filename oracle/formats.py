"""Scalar number formats, written from their published definitions (test infrastructure).

Formats and where their definition comes from:

* bf16 / fp32 — IEEE-754 binary formats (bf16 = fp32 with 7 fraction bits),
  round-to-nearest, ties to even.
* e4m3 — OCP 8-bit floating point "E4M3FN": 1 sign, 4 exponent (bias 7), 3 fraction
  bits, subnormals, no infinities, S.1111.111 is NaN, largest finite 448.
* e2m1 — OCP Microscaling v1.0 FP4: 1 sign, 2 exponent (bias 1), 1 fraction bit,
  values {0, 0.5, 1, 1.5, 2, 3, 4, 6}, no inf/NaN.
* E8M0 — OCP Microscaling v1.0 shared scale: an unsigned biased exponent, value
  2^(e-127), 0xFF is NaN.

Rounding is round-to-nearest-even everywhere ("satfinite" clamps out-of-range values
to the largest finite magnitude instead of overflowing). The quantization pages only
say "round" (explainer page, section "4비트 값에는 스케일이라는 해석 규칙이 붙는다");
RNE is the reading taken.

fp32 arithmetic is emulated in fp64 followed by one rounding to fp32; for a single
+, -, x or / of two fp32 operands this equals the correctly rounded fp32 result because
fp64 carries more than 2*24+2 significand bits (double rounding is innocuous).

Parity: pinned by exhaustive code tables, RNE tie cases and round trips in
tests/test_oracle_formats.py.
"""
import numpy as np

# (fraction bits, minimum normal exponent, largest finite value)
BF16 = (7, -126, (2.0 - 2.0 ** -7) * 2.0 ** 127)
FP32 = (23, -126, (2.0 - 2.0 ** -23) * 2.0 ** 127)
E4M3 = (3, -6, 448.0)
E2M1 = (1, 0, 6.0)


def round_to(x, fmt, satfinite=False):
    """Round float64 values to the nearest value of ``fmt`` (ties to even).

    Values whose rounding exceeds the largest finite value become +-inf, or the
    largest finite value when ``satfinite``. The sign of zero is kept.
    """
    frac_bits, emin, vmax = fmt
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, e = np.frexp(ax)                      # ax = m * 2**e with m in [0.5, 1)
    exp = np.maximum(e - 1, emin)            # floor(log2 ax), clamped into the subnormal range
    quantum = np.ldexp(1.0, exp - frac_bits)  # spacing of representable values at that exponent
    r = np.rint(ax / quantum) * quantum       # np.rint: round half to even; the division is exact
    over = r > vmax
    if satfinite:
        r = np.where(over, vmax, r)
    else:
        r = np.where(over, np.inf, r)
    return np.copysign(r, x)


def f32(x):
    """Round to fp32 (RNE), returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16r(x):
    """Round to bf16 (RNE, overflow to inf), returned as float64."""
    return round_to(x, BF16)


# ---------------------------------------------------------------- decoders (bit fields)

def decode_e2m1(code):
    """e2m1 code (0..15) -> value, from the bit fields."""
    c = np.asarray(code, dtype=np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m / 2.0, e - 1))
    return np.where(s == 1, -mag, mag)


def decode_e4m3(code):
    """e4m3 (E4M3FN) code (0..255) -> value; 0x7F and 0xFF decode to NaN."""
    c = np.asarray(code, dtype=np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def decode_e8m0(code):
    """E8M0 code (0..255) -> 2**(code-127); 0xFF decodes to NaN."""
    c = np.asarray(code, dtype=np.int64)
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, v)


def decode_bf16_bits(bits):
    """bf16 bit patterns (uint16) -> float64 values."""
    b = np.asarray(bits, dtype=np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- encoders (exact values -> codes)

def _encode_minifloat(v, exp_bits, frac_bits, bias):
    """Code of an exactly representable minifloat value (sign kept for -0)."""
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v).astype(np.int64)
    a = np.abs(v)
    emin = 1 - bias
    _, e = np.frexp(a)
    exp = e - 1
    normal = (a >= np.ldexp(1.0, emin))
    # normal: biased exponent and fraction; subnormal: exponent field 0, fraction = a / 2^(emin-frac)
    ef = np.where(normal, exp + bias, 0)
    frac = np.where(normal,
                    np.rint((a / np.ldexp(1.0, np.where(normal, exp, 0)) - 1.0) * (1 << frac_bits)),
                    np.rint(a / np.ldexp(1.0, emin - frac_bits)))
    code = (sign << (exp_bits + frac_bits)) | (ef.astype(np.int64) << frac_bits) | frac.astype(np.int64)
    back = _decode_generic(code, exp_bits, frac_bits, bias)
    if not np.array_equal(np.abs(back), a):
        raise ValueError("value not representable in the target format")
    return code


def _decode_generic(code, exp_bits, frac_bits, bias):
    c = np.asarray(code, dtype=np.int64)
    e = (c >> frac_bits) & ((1 << exp_bits) - 1)
    m = c & ((1 << frac_bits) - 1)
    mag = np.where(e == 0, np.ldexp(m / float(1 << frac_bits), 1 - bias),
                   np.ldexp(1.0 + m / float(1 << frac_bits), e - bias))
    s = (c >> (exp_bits + frac_bits)) & 1
    return np.where(s == 1, -mag, mag)


def encode_e2m1(v):
    """Exact e2m1 value -> 4-bit code."""
    return _encode_minifloat(v, 2, 1, 1).astype(np.uint8)


def encode_e4m3(v):
    """Exact finite e4m3 value -> 8-bit code."""
    return _encode_minifloat(v, 4, 3, 7).astype(np.uint8)


def e2m1_rne(x):
    """RNE to e2m1 with satfinite, returned as codes."""
    return encode_e2m1(round_to(x, E2M1, satfinite=True))


def e4m3_rne(x):
    """RNE to e4m3 with satfinite, returned as codes."""
    return encode_e4m3(round_to(x, E4M3, satfinite=True))


def bf16_bits(v):
    """Exact bf16 value (float64) -> uint16 bit pattern."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    if not np.array_equal(f.astype(np.float64), np.asarray(v, dtype=np.float64)):
        raise ValueError("value not representable in fp32")
    b = f.view(np.uint32)
    if np.any(b & np.uint32(0xFFFF)):
        raise ValueError("value not representable in bf16")
    return (b >> np.uint32(16)).astype(np.uint16)
