"""GPU parity of the W4A16 GEMM (INT4 g128 with/without zero-points, and MXFP4-W4A16)
through the C ABI, against the fp64 oracle with the tolerance
|Y - Yref| <= 1e-2*|Yref| + 1e-2*rms(Yref) per element."""
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


def run_case(hm, fmt, m, n, k, has_zero, seed=0):
    w = synth.weights(n, k, seed=seed)
    z = synth.zero_points(n, k // 128, seed=seed + 1) if has_zero else None
    qw = QuantWeight(fmt, w, z)
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=seed + 2)
    full, y = canary_out(m, n)
    hm.gemm(fmt, x.cuda(), packed, n, k, out=y)
    torch.cuda.synchronize()
    yref = og.gemm(bf16_np(x), qw.what)
    assert_close(y, yref, f"fmt={fmt} m={m} n={n} k={k} zp={has_zero}")
    check_canary(full, m, f"fmt={fmt} m={m} n={n} k={k}")
    assert hm.device_error() == 0


def test_tiny_config(hm):
    # 4 x 512 activations, 256 x 512 symmetric INT4 weights (seed 0)
    run_case(hm, 1, 4, 256, 512, False, seed=0)


@pytest.mark.parametrize("m", [1, 2, 7, 16, 17, 33, 64, 65, 128, 129, 300])
@pytest.mark.parametrize("has_zero", [False, True])
def test_int4_m_sweep(hm, m, has_zero):
    run_case(hm, 1, m, 384, 1024, has_zero, seed=m)


@pytest.mark.parametrize("m,n,k", [(3, 130, 256), (50, 258, 512), (257, 200, 384), (1, 128, 128)])
def test_int4_ragged(hm, m, n, k):
    run_case(hm, 1, m, n, k, True, seed=5)


@pytest.mark.parametrize("m", [1, 16, 100, 256])
def test_mxfp4_w4a16(hm, m):
    run_case(hm, 2, m, 256, 1024, False, seed=7)


@pytest.mark.parametrize("tile_m", ["16", "32", "64", "128", "192", "256"])
@pytest.mark.parametrize("stream_k", ["0", "1"])
def test_forced_configs(hm, env, tile_m, stream_k):
    env["HM_TILE_M"] = tile_m
    env["HM_STREAM_K"] = stream_k
    run_case(hm, 1, 70, 512, 2048, True, seed=9)
    if tile_m == "192":              # several token tiles, the last one ragged
        run_case(hm, 1, 450, 384, 1024, True, seed=10)


@pytest.mark.parametrize("fmt,m,n,k", [(1, 2048, 2560, 2560), (1, 2000, 2600, 2560), (2, 2304, 2560, 2560)])
def test_hybrid_waves(hm, env, fmt, m, n, k):
    """More whole 256-token tiles than SMs with HM_SK_HYBRID=1: the tiles a last partial wave would
    hold run first as stream-K ranges over every CTA (their partials handed to the owner), then the
    rest as whole tiles in full waves. Ragged M and N included; against the oracle, and
    bit-identical on repeat."""
    env["HM_SK_HYBRID"] = "1"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = hm.plan(fmt, m, n, k, sms)
    assert p["stream_k"] == 1 and 0 < p["sk_tiles"] < p["tiles"] and p["grid"] == sms, p
    w = synth.weights(n, k, seed=m)
    z = synth.zero_points(n, k // 128, seed=m + 1) if fmt == 1 else None
    qw = QuantWeight(fmt, w, z)
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=m + 2).cuda()
    ys = []
    for _ in range(2):
        full, y = canary_out(m, n)
        hm.gemm(fmt, x, packed, n, k, out=y)
        ys.append((full, y))
    torch.cuda.synchronize()
    assert_close(ys[0][1], og.gemm(bf16_np(x.cpu()), qw.what), f"hybrid fmt={fmt} m={m} n={n} k={k}")
    for full, _ in ys:
        check_canary(full, m, f"hybrid fmt={fmt} m={m}")
    assert torch.equal(ys[0][1], ys[1][1])
    assert hm.device_error() == 0


def test_repeated_calls_reuse_workspace(hm):
    """Stream-K counters return to zero, so a workspace serves many calls."""
    n, k, m = 1024, 4096, 8
    qw = QuantWeight(1, synth.weights(n, k, seed=3), synth.zero_points(n, k // 128, seed=4))
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=5)
    ws = hm.alloc_workspace(1, m, n, k)
    yref = og.gemm(bf16_np(x), qw.what)
    first = None
    for _ in range(3):
        y = hm.gemm(1, x.cuda(), packed, n, k, ws=ws)
        torch.cuda.synchronize()
        assert_close(y, yref, "repeat")
        if first is None:
            first = y.clone()
        else:
            assert torch.equal(first, y)      # deterministic split-K reduction


@pytest.mark.parametrize("n,k", [(14336, 4096), (4096, 4096), (4096, 14336)])
def test_full_size_sampled(hm, n, k):
    """The benchmark's three W4A16 layers at M = 1, 4096 (on 4096x14336 the leftover wave's tiles run
    as stream-K ranges) and 8192, checked on sampled outputs."""
    w = synth.weights(n, k, seed=1)
    z = synth.zero_points(n, k // 128, seed=2)
    q, s = oq.quant_int4(w, zeros=z)
    d = hm.desc(1, n, k, True)
    from .gpu_util import pack_nibbles, to_bf16
    packed = hm.transform(d, torch.from_numpy(pack_nibbles(q)).cuda(), to_bf16(s).cuda(),
                          torch.from_numpy(z).cuda())
    rng = np.random.default_rng(0)
    for m in (1, 4096, 8192):
        x = synth.activations(m, k, seed=3)
        y = hm.gemm(1, x.cuda(), packed, n, k)
        torch.cuda.synchronize()
        ms = rng.integers(0, m, size=256)
        ns = rng.integers(0, n, size=256)
        xs = bf16_np(x[torch.from_numpy(ms)])
        what = oq.dequant_int4(q[ns], s[ns], z[ns])
        ref = np.einsum("ik,ik->i", xs, what)
        got = bf16_np(y.cpu()[torch.from_numpy(ms), torch.from_numpy(ns)])
        ok = og.tolerance_ok(got, ref)
        assert ok.all(), f"M={m}: {int((~ok).sum())} sampled outputs outside tolerance"
    assert hm.device_error() == 0


@pytest.mark.parametrize("log2_gain", [-100, 14])
def test_mxfp4_extreme_scales(hm, log2_gain):
    """MXFP4 blocks whose E8M0 exponent is far from 127: E > 128 takes the table path,
    small E restores through bf16 subnormal codes; both must match the oracle."""
    n, k, m = 256, 512, 16
    w = synth.weights(n, k, seed=17) * np.float32(2.0 ** log2_gain)
    qw = QuantWeight(2, w)
    _, packed = qw.transform(hm)
    e = oq.quant_mxfp4(w)[1]
    assert (e > 128).any() if log2_gain > 0 else (e < 40).all()
    x = synth.activations(m, k, seed=18)
    y = hm.gemm(2, x.cuda(), packed, n, k)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"mxfp4 gain 2^{log2_gain}")


@pytest.mark.parametrize("small", ["0", "1"])
@pytest.mark.parametrize("m", [1, 5, 16, 17, 32])
def test_small_token_kernel_and_general_kernel(hm, env, small, m):
    """INT4 token tiles of 16 and 32 go to the small-token kernel (group scale applied to each
    block's fp32 partial sum); HM_F16_SMALL=0 keeps the general kernel. Both must match the oracle,
    with stream-K splitting tiles (grid > tiles) and without."""
    env["HM_F16_SMALL"] = small
    env["HM_GEMV"] = "0"          # M <= 16 would otherwise take the warp-MMA decode kernel
    run_case(hm, 1, m, 640, 3072, True, seed=40 + m)
    run_case(hm, 1, m, 256, 1024, False, seed=60 + m)


@pytest.mark.parametrize("stream_k", ["0", "1"])
def test_small_token_kernel_long_k(hm, env, stream_k):
    """Many 128-K blocks per tile: the block-accumulator ring and A slots wrap many times."""
    env["HM_STREAM_K"] = stream_k
    env["HM_GEMV"] = "0"
    run_case(hm, 1, 9, 384, 14336, True, seed=77)
