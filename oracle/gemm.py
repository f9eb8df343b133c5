"""Reference GEMMs in fp64 (test infrastructure).

What the path computes, after the explainer page "vLLM Humming은 4비트를 어떻게 계산하나",
section "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다": a linear layer is
Y[M,N] = X[M,K] * W^T with W stored as [N,K]; the quantized layer replaces W by its
restored (dequantized) value, and for the A8/A4 formats X by its quantized value. The
MoE section of the same page splits tokens by expert, so the grouped GEMM is one such
product per expert over that expert's contiguous rows.

Each function takes the dequantized operands (see oracle.quant) and forms the plain
definition Y[m,n] = sum_k xhat[m,k] * what[n,k] with a library fp64 matmul. There is
no blocking or reordering beyond that; output rounding to bf16 happens on the GPU only,
the comparison tolerance is applied by the tests.

Parity: pinned in tests/test_oracle_gemm.py (exact integer special case, brute-force
triple loop, transposition-sensitive shapes, MoE = stacked dense).
"""
import numpy as np

from . import quant


def gemm(xhat, what):
    """Y = xhat @ what^T in fp64; xhat [M,K], what [N,K]."""
    return np.asarray(xhat, dtype=np.float64) @ np.asarray(what, dtype=np.float64).T


def gemm_w4a16_int4(x, q, s, zeros=None):
    """bf16 activations x [M,K] times restored INT4 weights."""
    return gemm(x, quant.dequant_int4(q, s, zeros))


def gemm_w4a16_mxfp4(x, codes, e):
    return gemm(x, quant.dequant_mxfp4(codes, e))


def gemm_w4a16_mxint4(x, q, e):
    return gemm(x, quant.dequant_mxint4(q, e))


def gemm_w4a8_mxfp4(xq, s_tok, codes, e):
    """Y[m,n] = s_tok[m] * sum_k e4m3(xq[m,k]) * what[n,k] (per-token scale outside the sum)."""
    from .formats import decode_e4m3
    acc = gemm(decode_e4m3(xq), quant.dequant_mxfp4(codes, e))
    return acc * np.asarray(s_tok, dtype=np.float64)[:, None]


def gemm_w4a4_nvfp4(xc, xsb, gx, wc, wsb, gw):
    """Y = gX*gW * sum_blocks sbX*sbW * sum_k e2m1X*e2m1W, written as the product of the
    two restored matrices (scales are exact in fp64)."""
    return gemm(quant.dequant_nvfp4(xc, xsb, gx), quant.dequant_nvfp4(wc, wsb, gw))


def moe_gemm(x, offsets, what_per_expert):
    """Grouped GEMM over expert-sorted rows: rows offsets[e]:offsets[e+1] use expert e."""
    x = np.asarray(x, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    n = what_per_expert[0].shape[0]
    y = np.zeros((x.shape[0], n), dtype=np.float64)
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b] = gemm(x[a:b], what_per_expert[e])
    return y


def tolerance_ok(y, yref, rel=1e-2, abs_rms=1e-2):
    """|Y - Yref| <= rel*|Yref| + abs_rms*rms(Yref), element-wise."""
    y = np.asarray(y, dtype=np.float64)
    yref = np.asarray(yref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(yref ** 2))) if yref.size else 0.0
    bound = rel * np.abs(yref) + abs_rms * rms
    return np.abs(y - yref) <= bound
