"""Pins for the oracle's GEMMs (CPU only): an exact integer special case that reduces to
numpy's integer matmul, brute-force loops on tiny non-square shapes, the per-token scale
identity, and MoE = stacked dense."""
import numpy as np

from oracle import gemm as G
from oracle import quant as Q
from oracle.formats import decode_e4m3


def test_unit_scale_integer_case_is_exact_integer_matmul():
    rng = np.random.default_rng(0)
    m, n, k = 5, 7, 256
    q = rng.integers(-8, 8, size=(n, k))
    x = rng.integers(-4, 5, size=(m, k))
    s = np.ones((n, k // 128))
    y = G.gemm_w4a16_int4(x.astype(np.float64), q, s)
    np.testing.assert_array_equal(y, (x @ q.T).astype(np.float64))
    z = rng.integers(0, 16, size=(n, k // 128))
    qz = rng.integers(0, 16, size=(n, k))
    y = G.gemm_w4a16_int4(x.astype(np.float64), qz, s, z)
    np.testing.assert_array_equal(y, (x @ (qz - np.repeat(z, 128, axis=1)).T).astype(np.float64))


def _brute(x, w):
    m, k = x.shape
    n = w.shape[0]
    y = np.zeros((m, n))
    for i in range(m):
        for j in range(n):
            acc = 0.0
            for t in range(k):
                acc += float(x[i, t]) * float(w[j, t])
            y[i, j] = acc
    return y


def test_w4a16_brute_force_tiny():
    rng = np.random.default_rng(1)
    m, n, k = 3, 5, 128
    w = rng.standard_normal((n, k)) * 0.02
    x = rng.standard_normal((m, k))
    z = rng.integers(0, 16, size=(n, 1))
    q, s = Q.quant_int4(w, zeros=z)
    what = Q.dequant_int4(q, s, z)
    np.testing.assert_allclose(G.gemm_w4a16_int4(x, q, s, z), _brute(x, what), rtol=1e-12, atol=1e-12)
    # swapping the operand roles gives a different matrix (catches a transposed operand)
    assert G.gemm_w4a16_int4(x, q, s, z).shape == (m, n)


def test_w4a8_per_token_scale_identity():
    rng = np.random.default_rng(2)
    m, n, k = 4, 6, 64
    x = rng.standard_normal((m, k))
    w = rng.standard_normal((n, k)) * 0.02
    xq, st = Q.quant_fp8_per_token(x)
    codes, e = Q.quant_mxfp4(w)
    y = G.gemm_w4a8_mxfp4(xq, st, codes, e)
    xhat = decode_e4m3(xq) * st[:, None]
    np.testing.assert_allclose(y, _brute(xhat, Q.dequant_mxfp4(codes, e)), rtol=1e-12, atol=1e-14)


def test_w4a4_unit_scales_reduce_to_code_products():
    rng = np.random.default_rng(3)
    m, n, k = 3, 4, 32
    xc = rng.integers(0, 16, size=(m, k)).astype(np.uint8)
    wc = rng.integers(0, 16, size=(n, k)).astype(np.uint8)
    one = np.full((m, 2), 0x38, np.uint8)          # e4m3 1.0
    onew = np.full((n, 2), 0x38, np.uint8)
    from oracle.formats import decode_e2m1
    y = G.gemm_w4a4_nvfp4(xc, one, 1.0, wc, onew, 1.0)
    np.testing.assert_array_equal(y, decode_e2m1(xc) @ decode_e2m1(wc).T)
    y2 = G.gemm_w4a4_nvfp4(xc, one, 2.0, wc, onew, 0.25)
    np.testing.assert_array_equal(y2, y * 0.5)


def test_moe_is_stacked_dense():
    rng = np.random.default_rng(4)
    e, n, k = 4, 6, 128
    offsets = np.array([0, 3, 3, 7, 9])
    x = rng.standard_normal((9, k))
    ws = [rng.standard_normal((n, k)) for _ in range(e)]
    y = G.moe_gemm(x, offsets, ws)
    for i in range(e):
        a, b = offsets[i], offsets[i + 1]
        np.testing.assert_array_equal(y[a:b], x[a:b] @ ws[i].T)


def test_linearity_power_of_two():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 128))
    q, s = Q.quant_int4(rng.standard_normal((3, 128)) * 0.02)
    np.testing.assert_array_equal(G.gemm_w4a16_int4(2 * x, q, s), 2 * G.gemm_w4a16_int4(x, q, s))


def test_tolerance_rule():
    yref = np.array([1.0, -2.0, 0.0, 100.0])
    rms = np.sqrt(np.mean(yref ** 2))
    ok = G.tolerance_ok(yref + np.array([0.0, 0.02, 0.01 * rms, 2.0]), yref)
    np.testing.assert_array_equal(ok, [True, True, True, False])


def test_w4a16_mxint4_exact_integer_case_and_brute_force():
    # E8M0 code 127 is scale 1: the product is numpy's integer matmul of q; other codes scale
    # each 32-block of K by its power of two, checked against explicit loops
    rng = np.random.default_rng(7)
    m, n, k = 3, 5, 128
    q = rng.integers(-8, 8, size=(n, k))
    x = rng.integers(-4, 5, size=(m, k))
    e = np.full((n, k // 32), 127)
    np.testing.assert_array_equal(G.gemm_w4a16_mxint4(x.astype(np.float64), q, e), (x @ q.T).astype(np.float64))
    e = rng.integers(120, 131, size=(n, k // 32))
    w = np.array([[q[j, t] * 2.0 ** (int(e[j, t // 32]) - 127) for t in range(k)] for j in range(n)])
    np.testing.assert_array_equal(G.gemm_w4a16_mxint4(x.astype(np.float64), q, e), _brute(x, w))


def test_w4a16_mxfp4_against_typed_e2m1_values():
    # the e2m1 code table written out from the format definition (sign bit 3, then
    # 0, 0.5, 1, 1.5, 2, 3, 4, 6), independent of the oracle's decoder, and a loop GEMM
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    rng = np.random.default_rng(8)
    m, n, k = 2, 3, 64
    codes = rng.integers(0, 16, size=(n, k))
    e = rng.integers(124, 131, size=(n, k // 32))
    x = rng.integers(-3, 4, size=(m, k)).astype(np.float64)
    w = np.array([[table[codes[j, t]] * 2.0 ** (int(e[j, t // 32]) - 127) for t in range(k)] for j in range(n)])
    np.testing.assert_array_equal(G.gemm_w4a16_mxfp4(x, codes, e), _brute(x, w))
