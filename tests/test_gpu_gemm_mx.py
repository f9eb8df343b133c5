"""GPU parity of the block-scaled GEMMs (W4A8 MXFP4 x FP8 per token, W4A4 NVFP4) through
the C ABI, against the oracle with |Y - Yref| <= 1e-2*|Yref| + 1e-2*rms(Yref)."""
import os

import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import gemm as og
from oracle import quant as oq

from .gpu_util import QuantWeight, assert_close, bf16_np, canary_out, check_canary

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


@pytest.fixture
def env():
    saved = dict(os.environ)
    yield os.environ
    os.environ.clear()
    os.environ.update(saved)


def w4a8_case(hm, m, n, k, seed=0, explicit=False):
    qw = QuantWeight(3, synth.weights(n, k, seed=seed))
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=seed + 1, outlier_frac=0.01)
    xq, st = oq.quant_fp8_per_token(bf16_np(x))
    yref = og.gemm_w4a8_mxfp4(xq, st, qw.q, qw.s)
    full, y = canary_out(m, n)
    if explicit:
        gq, gs = hm.quant_act_fp8(x.cuda())
        hm.gemm(3, gq, packed, n, k, x_scale=gs, out=y)
    else:
        hm.gemm(3, x.cuda(), packed, n, k, out=y)
    torch.cuda.synchronize()
    assert_close(y, yref, f"w4a8 m={m} n={n} k={k}")
    check_canary(full, m, f"w4a8 m={m} n={n} k={k}")
    assert hm.device_error() == 0


def w4a4_case(hm, m, n, k, seed=0, explicit=False):
    qw = QuantWeight(4, synth.weights(n, k, seed=seed))
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=seed + 1)
    xc, xsb, gx = oq.quant_nvfp4(bf16_np(x))
    yref = og.gemm_w4a4_nvfp4(xc, xsb, gx, qw.q, qw.s, qw.g)
    full, y = canary_out(m, n)
    if explicit:
        gq, gs, gg = hm.quant_act_nvfp4(x.cuda())
        hm.gemm(4, gq, packed, n, k, x_scale=gs, x_global=gg, out=y)
    else:
        hm.gemm(4, x.cuda(), packed, n, k, out=y)
    torch.cuda.synchronize()
    assert_close(y, yref, f"w4a4 m={m} n={n} k={k}")
    check_canary(full, m, f"w4a4 m={m} n={n} k={k}")
    assert hm.device_error() == 0


@pytest.mark.parametrize("m", [1, 16, 17, 64, 100, 128, 129, 300])
def test_w4a8_m_sweep(hm, m):
    w4a8_case(hm, m, 384, 1024, seed=m)


def test_w4a8_explicit_activation_quant(hm):
    w4a8_case(hm, 40, 256, 512, seed=3, explicit=True)


def test_w4a8_ragged_n(hm):
    w4a8_case(hm, 5, 200, 768, seed=4)


@pytest.mark.parametrize("m", [1, 16, 40, 64, 128, 200, 300])
def test_w4a4_m_sweep(hm, m):
    w4a4_case(hm, m, 384, 1024, seed=m)


def test_w4a4_explicit_activation_quant(hm):
    w4a4_case(hm, 70, 256, 512, seed=5, explicit=True)


def test_w4a4_ragged_n(hm):
    w4a4_case(hm, 3, 130, 256, seed=6)


@pytest.mark.parametrize("stream_k", ["0", "1"])
def test_forced_stream_k(hm, env, stream_k):
    env["HM_STREAM_K"] = stream_k
    w4a8_case(hm, 20, 256, 2048, seed=8)
    w4a4_case(hm, 20, 256, 2048, seed=9)


@pytest.mark.parametrize("fmt,n,k", [(3, 18432, 7168), (3, 7168, 7168), (4, 8192, 8192)])
def test_full_size_sampled(hm, fmt, n, k):
    """The benchmark's block-scaled layers, checked on sampled outputs: W4A8 at M = 1, 16, 1024 and
    8192, W4A4 at the benchmark's M = 16, 128, 1024 and 8192."""
    w = synth.weights(n, k, seed=2)
    qw = QuantWeight(fmt, w)
    _, packed = qw.transform(hm)
    rng = np.random.default_rng(1)
    for m in ((1, 16, 1024, 8192) if fmt == 3 else (16, 128, 1024, 8192)):
        x = synth.activations(m, k, seed=3, outlier_frac=0.01 if fmt == 3 else 0.0)
        y = hm.gemm(fmt, x.cuda(), packed, n, k)
        torch.cuda.synchronize()
        ms = rng.integers(0, m, size=128)
        ns = rng.integers(0, n, size=128)
        xv = bf16_np(x)
        if fmt == 3:
            xq, st = oq.quant_fp8_per_token(xv[ms])
            from oracle.formats import decode_e4m3
            xhat = decode_e4m3(xq) * st[:, None]
        else:
            gx = oq.nvfp4_global_scale(xv)              # the tensor scale needs all of X
            xc, xsb, _ = oq.quant_nvfp4(xv[ms], g=gx)   # the 16-blocks are row-local
            xhat = oq.dequant_nvfp4(xc, xsb, gx)
        ref = np.einsum("ik,ik->i", xhat, qw.what[ns])
        got = bf16_np(y.cpu()[torch.from_numpy(ms), torch.from_numpy(ns)])
        ok = og.tolerance_ok(got, ref)
        assert ok.all(), f"fmt={fmt} M={m}: {int((~ok).sum())} sampled outputs outside tolerance"
