"""Pins for the oracle's quantizers (CPU only): the explainer page's worked INT4 example,
hand-computed closed forms, and invariants every correct quantizer satisfies."""
import json
import os

import numpy as np

from oracle import formats as F
from oracle import quant as Q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int4_worked_example.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_page_worked_example_quantize_restore():
    g = golden()
    q = int(Q.int4_code(g["w"], g["scale"]))
    assert q == g["q"]
    assert abs(float(Q.int4_restore(q, g["scale"])) - g["restored"]) < 1e-12


def test_page_worked_example_range_clamp():
    lo, hi = golden()["int4_range"]
    assert int(Q.int4_code(1.0, 0.1)) == hi          # 10 -> 7
    assert int(Q.int4_code(-1.0, 0.1)) == lo         # -10 -> -8
    assert int(Q.int4_code(0.74, 0.1)) == hi


def test_page_worked_example_dot_product():
    g = golden()
    w = np.array(g["dot_weights"])
    x = np.array(g["dot_activations"], dtype=np.float64)
    assert abs(float(w @ x) - g["dot_exact"]) < 1e-12
    what = Q.int4_restore(Q.int4_code(w, g["scale"]), g["scale"])
    np.testing.assert_allclose(what, g["dot_quantized_weights"], atol=1e-12)
    assert abs(float(what @ x) - g["dot_after_quantization"]) < 1e-12


def _group(vals):
    w = np.zeros((1, 128), dtype=np.float64)
    w[0, :len(vals)] = vals
    return w


def test_int4_symmetric_closed_form():
    # amax 0.875 -> s = 0.875/7 = 0.125 exactly -> q = w/0.125
    w = _group([0.875, -0.5, 0.125, 0.0, 0.3125, -0.0625])
    q, s = Q.quant_int4(w)
    assert s.shape == (1, 1) and s[0, 0] == 0.125
    np.testing.assert_array_equal(q[0, :6], [7, -4, 1, 0, 2, 0])   # 2.5 -> 2, -0.5 -> -0 (even)
    np.testing.assert_array_equal(Q.dequant_int4(q, s)[0, :6], [0.875, -0.5, 0.125, 0, 0.25, 0])


def test_int4_zero_point_closed_form():
    w = _group([0.875, -0.5, 0.125, 0.0])
    z = np.array([[3]])
    q, s = Q.quant_int4(w, zeros=z)
    np.testing.assert_array_equal(q[0, :4], [10, 0, 4, 3])           # -4+3 = -1 clamps to 0
    np.testing.assert_array_equal(Q.dequant_int4(q, s, z)[0, :4], [0.875, -0.375, 0.125, 0])


def test_int4_scale_is_bf16_of_fp32_quotient():
    w = _group([0.7])
    _, s = Q.quant_int4(w)
    want = F.bf16r(np.float64(np.float32(np.float32(0.7) / np.float32(7.0))))
    assert s[0, 0] == want and s[0, 0] != 0.1


def test_int4_zero_group():
    q, s = Q.quant_int4(np.zeros((2, 256)))
    assert np.all(s == 0) and np.all(q == 0)
    q, s = Q.quant_int4(np.zeros((1, 128)), zeros=np.array([[5]]))
    assert np.all(q == 5)


def test_int4_invariants_random():
    rng = np.random.default_rng(0)
    w = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    q, s = Q.quant_int4(w)
    assert q.min() >= -7 and q.max() <= 7              # s = amax/7 never reaches -8
    sf = np.repeat(s, 128, axis=1)
    err = np.abs(w - q * sf)
    assert np.all(err <= sf * (0.5 + 1e-3))            # round-to-nearest bound (bf16 scale)
    g = np.abs(w.reshape(64, 4, 128))
    arg = g.argmax(axis=2)
    qmax = np.take_along_axis(np.abs(q.reshape(64, 4, 128)), arg[..., None], axis=2)
    assert np.all(qmax == 7)


def test_int4_zero_point_invariants_random():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((32, 256)) * 0.02).astype(np.float32)
    z = rng.integers(0, 16, size=(32, 2))
    q, s = Q.quant_int4(w, zeros=z)
    assert q.min() >= 0 and q.max() <= 15
    sf = np.repeat(s, 128, axis=1)
    zf = np.repeat(z, 128, axis=1)
    inside = (q > 0) & (q < 15)
    err = np.abs(w - (q - zf) * sf)
    assert np.all(err[inside] <= sf[inside] * (0.5 + 1e-3))
    # clamped entries moved towards the range edge
    assert np.all(w[q == 0] / sf[q == 0] - (0 - zf[q == 0]) <= 0.5 + 1e-3)


def test_mxfp4_scale_rule_closed_forms():
    def one(amax_val, probe):
        w = np.zeros((1, 32))
        w[0, 0] = amax_val
        w[0, 1] = probe
        codes, e = Q.quant_mxfp4(w)
        return int(e[0, 0]), int(codes[0, 0]), int(codes[0, 1])
    assert one(6.0, 0.0) == (127, 7, 0)        # floor(log2 6) = 2 -> 2-2+127
    assert one(5.0, 0.75) == (127, 6, 2)       # 5 is a tie between 4 and 6 -> 4; 0.75 -> 1
    assert one(12.0, -3.0) == (128, 7, 0xB)    # scale 2: 12/2 = 6, -3/2 = -1.5
    assert one(0.1, 0.0) == (121, 7, 0)        # 0.1 * 2^6 = 6.4 saturates to 6
    codes, e = Q.quant_mxfp4(np.zeros((1, 32)))
    assert e[0, 0] == 0 and np.all(codes == 0)


def test_mxfp4_invariants_random():
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((16, 256)) * 0.02).astype(np.float32)
    codes, e = Q.quant_mxfp4(w)
    what = Q.dequant_mxfp4(codes, e)
    scale = np.repeat(F.decode_e8m0(e), 32, axis=1)
    mags = np.abs(F.decode_e2m1(codes))
    assert mags.max() <= 6
    # the block maximum lands on 4 or 6 (amax / 2^(floor(log2 amax)-2) is in [4, 8))
    blk = np.abs(w.reshape(16, 8, 32)).argmax(axis=2)
    top = np.take_along_axis(mags.reshape(16, 8, 32), blk[..., None], axis=2)
    assert set(np.unique(top)) <= {4.0, 6.0}
    # error of RNE on the e2m1 grid: at most half the local spacing (1 above 2, 2 above 4)
    r = np.abs(w) / scale
    spacing = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))
    assert np.all(np.abs(w - what) <= scale * spacing / 2 + scale * np.maximum(r - 6, 0) + 1e-12)


def test_fp8_per_token_closed_form():
    x = np.array([[448.0, -1.0, 0.5, 0.0], [0.0, 0.0, 0.0, 0.0], [2.0, 1.0, -0.5, 0.25]])
    xq, s = Q.quant_fp8_per_token(x)
    np.testing.assert_array_equal(s, [1.0, 0.0, np.float32(2.0 / 448.0)])
    np.testing.assert_array_equal(xq[0], [0x7E, 0xB8, 0x30, 0x00])
    assert np.all(xq[1] == 0)
    assert xq[2, 0] == 0x7E                           # the row maximum maps to 448


def test_fp8_per_token_invariants_random():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((8, 1024)).astype(np.float32)
    x = x.astype(np.float64)
    xq, s = Q.quant_fp8_per_token(x)
    back = Q.dequant_fp8_per_token(xq, s)
    big = np.abs(x) > 2.0 ** -6 * s[:, None] * 448 / 448  # normal range of e4m3 after scaling
    rel = np.abs(back - x)[big] / np.abs(x)[big]
    assert rel.max() <= 2.0 ** -4 + 1e-6                # 3 fraction bits: half-ulp relative
    assert np.all(np.abs(F.decode_e4m3(xq)).max(axis=1) == 448)


def test_nvfp4_closed_form():
    # tensor amax 2688 -> g = 1; block amax 6 -> sb = 1 (code 0x38)
    v = np.zeros((1, 32))
    v[0, 0] = 2688.0
    v[0, 16:20] = [6.0, -3.0, 1.0, 0.25]
    codes, sb, g = Q.quant_nvfp4(v)
    assert g == 1.0
    assert sb[0, 1] == 0x38
    np.testing.assert_array_equal(codes[0, 16:20], [7, 0xD, 2, 0])
    assert sb[0, 0] == 0x7E and codes[0, 0] == 7      # 2688/6 = 448 -> element 6
    c, s2, g2 = Q.quant_nvfp4(np.zeros((2, 16)))
    assert g2 == 1.0 and np.all(s2 == 0) and np.all(c == 0)


def test_nvfp4_invariants_random():
    rng = np.random.default_rng(4)
    v = (rng.standard_normal((16, 256)) * 0.02).astype(np.float32)
    codes, sb, g = Q.quant_nvfp4(v)
    assert g == np.float32(np.abs(v).max() / np.float32(2688.0))
    back = Q.dequant_nvfp4(codes, sb, g)
    scale = np.repeat(F.decode_e4m3(sb), 16, axis=1) * g
    assert np.all(np.abs(back - v) <= scale * 1.0 + 1e-12)  # half of the widest e2m1 gap (2)


# ------------------------------------------------------------------ MXINT4

def test_mxint4_scale_rule_closed_forms():
    def one(amax_val, probe):
        w = np.zeros((1, 32))
        w[0, 0] = amax_val
        w[0, 1] = probe
        q, e = Q.quant_mxint4(w)
        return int(e[0, 0]), int(q[0, 0]), int(q[0, 1])
    assert one(1.0, 0.3) == (125, 4, 1)          # X = 1/4: 1 -> 4, 0.3 -> rne(1.2) = 1
    assert one(7.0, -2.0) == (127, 7, -2)        # floor(log2 7) = 2: X = 1
    assert one(8.0, 3.0) == (128, 4, 2)          # X = 2: 3/2 = 1.5 is a tie -> 2
    assert one(0.3, 0.03125) == (123, 5, 0)      # X = 1/16: 4.8 -> 5; 0.5 is a tie -> 0
    assert one(-1.875, 1.875) == (125, -8, 7)    # -7.5 -> -8 (even); +7.5 -> 8 clamps to 7
    assert one(1.9375, -1.9375) == (125, 7, -8)  # 7.75 -> 8 clamps to 7; -7.75 -> -8
    q, e = Q.quant_mxint4(np.zeros((1, 32)))
    assert e[0, 0] == 0 and np.all(q == 0) and np.all(Q.dequant_mxint4(q, e) == 0)


def test_mxint4_codes_brute_force():
    # each code is the integer in [-8, 7] nearest to w / X, ties to the even one, found by
    # scanning all sixteen candidates
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((6, 128)) * rng.choice([0.01, 1.0, 300.0], size=(6, 1))).astype(np.float32)
    w[0, :32] = np.array([(c + 0.5) / 4 for c in range(-8, 8)] * 2, dtype=np.float32)   # exact ties
    q, e = Q.quant_mxint4(w)
    x = F.decode_e8m0(e)
    cand = np.arange(-8, 8)
    for r in range(w.shape[0]):
        for c in range(w.shape[1]):
            v = float(w[r, c]) / float(x[r, c // 32])
            d = np.abs(v - cand)
            best = cand[d == d.min()]
            want = best[0] if len(best) == 1 else best[best % 2 == 0][0]
            assert q[r, c] == want, (r, c, v)


def test_mxint4_invariants_random():
    rng = np.random.default_rng(12)
    w = (rng.standard_normal((16, 256)) * 0.02).astype(np.float32)
    q, e = Q.quant_mxint4(w)
    what = Q.dequant_mxint4(q, e)
    scale = np.repeat(F.decode_e8m0(e), 32, axis=1)
    assert q.min() >= -8 and q.max() <= 7
    # the block maximum lands on a magnitude in [4, 8] (amax / X is in [4, 8))
    top = np.abs(q).reshape(16, 8, 32).max(axis=2)
    assert top.min() >= 4 and top.max() <= 8
    # round-to-nearest error, plus the clamp of values above 7.5 X to 7 X
    r = w / scale
    assert np.all(np.abs(w - what) <= scale / 2 + scale * np.maximum(r - 7.5, 0) + 1e-12)
    # restored values are bf16 numbers (at most four significant bits times a power of two)
    np.testing.assert_array_equal(F.bf16r(what), what)


def test_mxint4_exact_on_its_own_grid():
    # weights that are q * 2^j with the block's largest |q| in [4, 7] come back unchanged
    rng = np.random.default_rng(13)
    q0 = rng.integers(-7, 8, size=(4, 64))
    q0[:, 0], q0[:, 32] = 7, -5
    j = np.array([[-20, 3], [0, -1], [10, -7], [-3, 5]])
    w = q0 * np.ldexp(1.0, np.repeat(j, 32, axis=1))
    q, e = Q.quant_mxint4(w)
    np.testing.assert_array_equal(q, q0)
    np.testing.assert_array_equal(e, j + 127)
    np.testing.assert_array_equal(Q.dequant_mxint4(q, e), w)


def test_nvfp4_hand_computed_tensor_scale_not_one():
    """A row with tensor amax 1, so g = fp32(1/2688) = 0x39C30C31 (3.7202382e-4), not 1.

    Every value is an fp32 bit pattern chosen at a rounding boundary, so that another order of
    the recipe's fp32 steps gives other codes: sb from the exact amax/(6g), or from
    amax/fp32(6g), or amax*fp32(1/(6g)); elements divided by the exact sb*g instead of its fp32
    rounding, or by g then sb, or by sb then g, or multiplied by the fp32 reciprocal of fp32(sb*g).
    The steps, worked by hand in exact arithmetic (fp32 rounding after each operation):

    block 0: amax 1: fp32(1/6) = 0.16666667163, /g -> 448.0 (e4m3 0x7E); d = fp32(448*g) =
             0.16666667163; 1/d = 6.0 -> e2m1 6 (code 7).
    block 1: amax 0x3B76DB6D = 0.0037667409: fp32(amax/6) = 6.2779017e-4, /g = 1.6875 exactly, the
             e4m3 midpoint of 1.625 and 1.75, ties to even -> 1.75 (0x3E) (the exact quotient is
             just below 1.6875 -> 1.625); d = fp32(1.75*g) = 6.5104169e-4 (rounded up).
             0x392AAAAB = d/4 exactly: v/d = 0.25, tie -> 0 (code 0) (exact sb*g < d: 0.5);
             0x3A955555: v/d = 1.7499999 -> 1.5 (code 3) (times fp32(1/d): 1.75 -> 2);
             0x3A000000: v/d rounds to 0.75 in fp32, a tie -> 1.0 (code 2) (the exact quotient
             by sb*g is just below 0.75 -> 0.5); -0x3A955555 -> code 11; amax/d = 5.79 -> 6
             (code 7).
    block 2: amax 0x3B400001 = 0.0029296877: fp32(amax/6)/g = 1.3125001 -> 1.375 (0x3B)
             (amax/fp32(6g) = 1.3124999 -> 1.25); d = 5.1153277e-4.
             0x39C92492: v/d = 0.74999994 -> 0.5 (code 1) (fp32(v/g)/sb: 0.75 -> 1.0);
             0x3A279E7B: v/d = 1.25, tie -> 1.0 (code 2) (exact, v/g/sb and v/sb/g: 1.5);
             its negative -> code 10.
    block 3: amax 0x3B2DB6DB = 0.0026506695: fp32(amax/6)/g = 1.1874999 -> 1.125 (0x39)
             (amax*fp32(1/(6g)): 1.1875 -> 1.25); +-amax/d = +-6.333 -> +-6 (codes 7, 15).
    """
    def f(h):
        return float(np.array([h], dtype=np.uint32).view(np.float32)[0])
    v = np.zeros((1, 64))
    v[0, 0] = 1.0
    v[0, 16:21] = [f(0x3B76DB6D), f(0x392AAAAB), f(0x3A955555), f(0x3A000000), -f(0x3A955555)]
    v[0, 32:36] = [f(0x3B400001), f(0x39C92492), f(0x3A279E7B), -f(0x3A279E7B)]
    v[0, 48:50] = [f(0x3B2DB6DB), -f(0x3B2DB6DB)]
    codes, sb, g = Q.quant_nvfp4(v)
    assert np.float32(g).view(np.uint32) == 0x39C30C31
    assert list(sb[0]) == [0x7E, 0x3E, 0x3B, 0x39]
    expect = np.zeros(64, dtype=np.int64)
    expect[0] = 7
    expect[16:21] = [7, 0, 3, 2, 11]
    expect[32:36] = [7, 1, 2, 10]
    expect[48:50] = [7, 15]
    np.testing.assert_array_equal(codes[0], expect)
    # restored values: e2m1 * sb * g
    back = Q.dequant_nvfp4(codes, sb, g)
    assert back[0, 18] == 1.5 * 1.75 * g and back[0, 49] == -6.0 * 1.125 * g


def test_gptq_zero_convention():
    # symmetric 4-bit quantization has z = 8, which GPTQ-style checkpoints store as 7; z = 0 wraps to
    # 15; every z in [0, 15] comes back from its stored value
    assert int(Q.gptq_stored_zero(8)) == 7 and int(Q.gptq_stored_zero(0)) == 15 and int(Q.gptq_stored_zero(15)) == 14
    z = np.arange(16)
    np.testing.assert_array_equal(Q.zero_from_gptq(Q.gptq_stored_zero(z)), z)
    assert sorted(Q.gptq_stored_zero(z).tolist()) == list(range(16))     # a bijection on four bits


def test_int4_wide_groups_and_per_channel():
    # a group of 256 is one scale over two 128-blocks: s = bf16(max|w| / 7) over all 256 values
    rng = np.random.default_rng(12)
    w = rng.standard_normal((3, 512)).astype(np.float32)
    w[1, 300] = 9.0                                     # the second group of row 1
    q, s = Q.quant_int4(w, group=256)
    assert s.shape == (3, 2)
    assert s[1, 1] == F.bf16r(np.float32(9.0) / np.float32(7.0)) and q[1, 300] == 7
    # per channel: one scale per row
    q1, s1 = Q.quant_int4(w, group=512)
    assert s1.shape == (3, 1) and s1[1, 0] == s[1, 1]
    back = Q.dequant_int4(q1, s1, group=512)
    # half a step of the row's scale, plus the bf16 rounding of the restored value
    assert np.all(np.abs(back - w) <= np.repeat(s1, 512, axis=1) * 0.5 + 2.0 ** -8 * np.abs(w) + 1e-6)


def test_int8_closed_forms():
    # one group of 128 with max |w| = 1.27: s = bf16(1.27 / 127) = bf16(0.01) = 0.010009765625
    w = np.zeros((1, 128))
    w[0, :4] = [1.27, -0.5, 0.005004882812, -1.3]
    q, s = Q.quant_int8(w)
    assert s[0, 0] == F.bf16r(np.float32(1.3) / np.float32(127.0))
    sv = s[0, 0]
    assert q[0, 3] == -127 and q[0, 0] == int(np.rint(np.float32(1.27) / np.float32(sv)))
    # range: -128 appears only through clamping, +127 at the group maximum
    assert q.min() >= -128 and q.max() <= 127
    # zero-points: q + z, clamped into [0, 255]
    qz, _ = Q.quant_int8(w, zeros=np.array([[200]]))
    assert qz[0, 3] == 200 - 127 and qz[0, 0] == min(200 + q[0, 0], 255)
    back = Q.dequant_int8(qz, s, np.array([[200]]))
    assert back[0, 1] == F.bf16r((qz[0, 1] - 200) * sv)


def test_int8_brute_force():
    # every code is the integer in range nearest to fp32(w / s), ties to even, by scanning all candidates
    rng = np.random.default_rng(13)
    w = (rng.standard_normal((3, 256)) * 0.05).astype(np.float32)
    z = np.array([[0, 255], [128, 7], [60, 200]])
    for zeros in (None, z):
        q, s = Q.quant_int8(w, zeros=zeros)
        for r in range(3):
            for c in range(0, 256, 7):
                sv = float(s[r, c // 128])
                quot = float(np.float32(np.float32(w[r, c]) / np.float32(sv)))
                zz = 0 if zeros is None else int(zeros[r, c // 128])
                lo, hi = (-128, 127) if zeros is None else (0, 255)
                cands = np.arange(lo, hi + 1)
                d = np.abs(cands - zz - quot)
                best = cands[d == d.min()]
                pick = best[0] if len(best) == 1 else [b for b in best if (b - zz) % 2 == 0][0]
                assert q[r, c] == pick
