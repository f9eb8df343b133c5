"""GPU parity of the warp-MMA W4A16 kernel for decode-sized M (1..32 tokens), through the C ABI,
against the fp64 oracle with the tolerance |Y - Yref| <= 1e-2*|Yref| + 1e-2*rms(Yref).

The kernel splits the packed 128x128 units over the CTAs; the shapes below cover tiles shared by
many CTAs (the last-arriving warp sums the partials), tiles owned whole by one CTA, CTAs whose
range spans several tiles, ragged N, single-block K and long K."""
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


def quantized(hm, fmt, n, k, has_zero, seed):
    w = synth.weights(n, k, seed=seed)
    z = synth.zero_points(n, k // 128, seed=seed + 1) if has_zero else None
    qw = QuantWeight(fmt, w, z)
    _, packed = qw.transform(hm)
    return qw, packed


def check(hm, fmt, m, n, k, has_zero, seed):
    qw, packed = quantized(hm, fmt, n, k, has_zero, seed)
    x = synth.activations(m, k, seed=seed + 2)
    # INT4 at 17..32 tokens takes the decode kernel only where tcgen05 would split tiles; force it
    saved = os.environ.get("HM_GEMV")
    os.environ["HM_GEMV"] = "2"
    os.environ["HM_DECODE_TC"] = "0"   # INT4 up to 16 tokens: the warp-MMA kernel, not the tensor-core one
    try:
        p = hm.plan(fmt, m, n, k, torch.cuda.get_device_properties(0).multi_processor_count)
        assert p["kernel"] == 1 and p["tile_m"] >= m
        full, y = canary_out(m, n)
        hm.gemm(fmt, x.cuda(), packed, n, k, out=y)
        torch.cuda.synchronize()
    finally:
        del os.environ["HM_DECODE_TC"]
        if saved is None:
            del os.environ["HM_GEMV"]
        else:
            os.environ["HM_GEMV"] = saved
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"fmt={fmt} m={m} n={n} k={k} zp={has_zero}")
    check_canary(full, m, f"decode m={m} n={n} k={k}")
    assert hm.device_error() == 0
    return p


# (n, k): 5 tiles each cut into 24 K ranges (global hand-off) | 2 units, no split, ragged N |
# 152 tiles of 2 blocks: one whole tile per CTA | 32 tiles cut into 4 ranges (clusters of 4) |
# 2 tiles x 112 blocks cut into 76 ranges | 64 tiles cut in 2 (clusters of 2) | 40 tiles cut in 3 |
# 160 tiles > 152 SMs: ranges of ~8.4 units run across tiles (a CTA publishes one shared tile and
# owns another, several segment ends per CTA)
SHAPES = [(640, 3072), (200, 128), (19456, 256), (4096, 4096), (256, 14336), (8192, 1024), (5120, 1024),
          (20480, 1024)]


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 15, 16, 17, 24, 31, 32])
@pytest.mark.parametrize("n,k", SHAPES)
def test_int4_zero_point(hm, m, n, k):
    check(hm, 1, m, n, k, True, seed=100 + m)


@pytest.mark.parametrize("m", [1, 3, 8, 11, 16, 20, 32])
@pytest.mark.parametrize("n,k", SHAPES)
def test_int4_symmetric(hm, m, n, k):
    check(hm, 1, m, n, k, False, seed=200 + m)


@pytest.mark.parametrize("m", [1, 2, 4, 6, 8, 10, 16, 25, 32])
@pytest.mark.parametrize("n,k", SHAPES)
def test_mxfp4(hm, m, n, k):
    check(hm, 2, m, n, k, False, seed=300 + m)


@pytest.mark.parametrize("log2_gain", [-100, 14])
@pytest.mark.parametrize("m", [1, 5, 13, 29])
def test_mxfp4_extreme_scales(hm, m, log2_gain):
    """E8M0 exponents above 128 take the fp32 restore, tiny ones bf16 subnormal codes."""
    n, k = 256, 512
    w = synth.weights(n, k, seed=17) * np.float32(2.0 ** log2_gain)
    qw = QuantWeight(2, w)
    _, packed = qw.transform(hm)
    e = oq.quant_mxfp4(w)[1]
    assert (e > 128).any() if log2_gain > 0 else (e < 40).all()
    x = synth.activations(m, k, seed=18)
    y = hm.gemm(2, x.cuda(), packed, n, k)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"mxfp4 gain 2^{log2_gain}")
    assert hm.device_error() == 0


@pytest.mark.parametrize("m", [1, 8, 16, 32])
def test_deterministic_and_workspace_reuse(hm, m):
    """The last-arriver hand-off sums partials in CTA order and clears its counters: repeated calls
    on one workspace, and a fresh workspace, give bit-identical outputs."""
    n, k = 4096, 4096
    qw, packed = quantized(hm, 1, n, k, True, seed=400 + m)
    x = synth.activations(m, k, seed=401).cuda()
    ws = hm.alloc_workspace(1, m, n, k)
    ys = [hm.gemm(1, x, packed, n, k, ws=ws).clone() for _ in range(4)]
    ys.append(hm.gemm(1, x, packed, n, k))
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(ys[0], y)
    assert_close(ys[0], og.gemm(bf16_np(x.cpu()), qw.what), "repeat")
    assert hm.device_error() == 0


@pytest.mark.parametrize("m", [1, 3, 8, 16, 32])
def test_tensor_core_path_still_matches(hm, env, m):
    """HM_GEMV=0 keeps the tcgen05 kernels for M <= 32: both paths agree with the oracle."""
    n, k = 640, 3072
    qw, packed = quantized(hm, 1, n, k, True, seed=500 + m)
    x = synth.activations(m, k, seed=501)
    env["HM_GEMV"] = "0"
    p = hm.plan(1, m, n, k, torch.cuda.get_device_properties(0).multi_processor_count)
    assert p["kernel"] == 0
    y_tc = hm.gemm(1, x.cuda(), packed, n, k)
    env["HM_GEMV"] = "1"
    y_mma = hm.gemm(1, x.cuda(), packed, n, k)
    torch.cuda.synchronize()
    ref = og.gemm(bf16_np(x), qw.what)
    assert_close(y_tc, ref, "tcgen05")
    assert_close(y_mma, ref, "warp-MMA decode kernel")
    assert hm.device_error() == 0


def test_full_size_sampled(hm):
    """The 14336 x 4096 layer at M = 1, 8, 16 and 32, checked on sampled outputs."""
    n, k = 14336, 4096
    w = synth.weights(n, k, seed=1)
    z = synth.zero_points(n, k // 128, seed=2)
    q, s = oq.quant_int4(w, zeros=z)
    d = hm.desc(1, n, k, True)
    from .gpu_util import pack_nibbles, to_bf16
    packed = hm.transform(d, torch.from_numpy(pack_nibbles(q)).cuda(), to_bf16(s).cuda(),
                          torch.from_numpy(z).cuda())
    rng = np.random.default_rng(0)
    for m in (1, 8, 16, 32):
        x = synth.activations(m, k, seed=3)
        y = hm.gemm(1, x.cuda(), packed, n, k)
        torch.cuda.synchronize()
        ms = rng.integers(0, m, size=512)
        ns = rng.integers(0, n, size=512)
        xs = bf16_np(x[torch.from_numpy(ms)])
        ref = np.einsum("ik,ik->i", xs, oq.dequant_int4(q[ns], s[ns], z[ns]))
        got = bf16_np(y.cpu()[torch.from_numpy(ms), torch.from_numpy(ns)])
        ok = og.tolerance_ok(got, ref)
        assert ok.all(), f"M={m}: {int((~ok).sum())} sampled outputs outside tolerance"
    assert hm.device_error() == 0


@pytest.mark.parametrize("n,k,m", [(4096, 4096, 1), (8192, 1024, 8), (5120, 1024, 16), (4096, 14336, 3), (4096, 4096, 32)])
def test_cluster_and_global_handoff_agree(hm, n, k, m):
    """Tiles cut into 2-4 K ranges are summed through a thread-block cluster's shared memory, or
    (HM_GEMV_CLUSTER=0, read once per process: run in a child) through global memory; both add the
    ranges in the same order, so the outputs are bit-identical."""
    import subprocess, sys, tempfile, textwrap
    qw, packed = quantized(hm, 1, n, k, True, seed=600 + m)
    x = synth.activations(m, k, seed=601)
    y = hm.gemm(1, x.cuda(), packed, n, k)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), "cluster hand-off")
    with tempfile.TemporaryDirectory() as d:
        torch.save({"packed": packed.cpu(), "x": x}, d + "/in.pt")
        code = textwrap.dedent(f"""
            import torch, __graft_entry__
            from moe_hm_gemm_gb300 import hm
            t = torch.load("{d}/in.pt")
            y = hm.gemm(1, t["x"].cuda(), t["packed"].cuda(), {n}, {k})
            torch.cuda.synchronize()
            assert hm.device_error() == 0
            torch.save(y.cpu(), "{d}/y.pt")
        """)
        env = dict(os.environ, HM_GEMV_CLUSTER="0")
        subprocess.run([sys.executable, "-c", code], check=True, env=env, cwd=os.getcwd())
        y_global = torch.load(d + "/y.pt")
    assert torch.equal(y.cpu(), y_global)
    assert hm.device_error() == 0
