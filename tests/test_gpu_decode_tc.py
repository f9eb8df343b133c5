"""GPU parity of the tensor-core decode kernel (INT4 weights, up to 16 tokens, restored weights in
TMEM as the tcgen05 MMA's A operand; selected with HM_DECODE_TC=1) against the oracle: every M up to 16, zero-points or not, tiles
cut along K between CTAs (fixed-owner hand-off), ranges across tiles, ragged N, a single 128-K
block, an odd number of k-blocks (load stages straddling two tiles), determinism, and agreement with
the warp-MMA decode kernel."""
import os

import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import gemm as og

from .gpu_util import QuantWeight, assert_close, bf16_np, canary_out, check_canary

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


@pytest.fixture(autouse=True)
def tensor_core_decode(monkeypatch):
    """The planner takes the tensor-core decode kernel only when asked to (HM_DECODE_TC=1)."""
    monkeypatch.setenv("HM_DECODE_TC", "1")


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def weight(hm, n, k, has_zero, seed):
    z = synth.zero_points(n, k // 128, seed=seed + 1) if has_zero else None
    qw = QuantWeight(1, synth.weights(n, k, seed=seed), z)
    return qw, qw.transform(hm)[1]


def run(hm, qw, packed, m, n, k, seed):
    p = hm.plan(1, m, n, k, sms())
    assert p["kernel"] == 2 and p["tile_m"] == 16, p
    x = synth.activations(m, k, seed=seed)
    full, y = canary_out(m, n)
    hm.gemm(1, x.cuda(), packed, n, k, out=y)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"decode-tc m={m} n={n} k={k}")
    check_canary(full, m, f"decode-tc m={m} n={n} k={k}")
    assert hm.device_error() == 0
    return x, y


# (n, k): 5 tiles cut into 24 K ranges | 160 tiles over the SMs (ranges across tiles) | ragged N,
# one unit | 7 k-blocks per tile (stages straddle tiles) | the benchmark's 4096 x 4096 layer
SHAPES = [(640, 3072), (20480, 1024), (200, 128), (384, 896), (4096, 4096)]


@pytest.mark.parametrize("m", [1, 2, 3, 5, 8, 9, 12, 15, 16])
@pytest.mark.parametrize("n,k", SHAPES)
def test_int4_zero_points(hm, m, n, k):
    qw, packed = weight(hm, n, k, True, seed=7 * m + n)
    run(hm, qw, packed, m, n, k, seed=m)


@pytest.mark.parametrize("m", [1, 7, 16])
@pytest.mark.parametrize("n,k", SHAPES)
def test_int4_symmetric(hm, m, n, k):
    qw, packed = weight(hm, n, k, False, seed=11 * m + k)
    run(hm, qw, packed, m, n, k, seed=100 + m)


def test_deterministic_and_agrees_with_warp_mma_kernel(hm, monkeypatch):
    """Two calls give identical bits (split tiles summed in CTA order); the warp-MMA decode kernel
    (which scales each 128-K block's exact sum instead of each weight) agrees within the tolerance."""
    n, k, m = 640, 3072, 6
    qw, packed = weight(hm, n, k, True, seed=3)
    x, y1 = run(hm, qw, packed, m, n, k, seed=4)
    y2 = hm.gemm(1, x.cuda(), packed, n, k)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    monkeypatch.setenv("HM_DECODE_TC", "0")
    assert hm.plan(1, m, n, k, sms())["kernel"] == 1
    y3 = hm.gemm(1, x.cuda(), packed, n, k)
    torch.cuda.synchronize()
    assert_close(y3, og.gemm(bf16_np(x), qw.what), "warp-MMA decode")
    assert hm.device_error() == 0


def test_mismatched_header_stores_nothing(hm):
    n, k = 256, 512
    qw, packed = weight(hm, n, 2 * k, False, seed=5)   # made for another K
    x = synth.activations(4, k, seed=6).cuda()
    y = torch.full((4, n), 7.0, dtype=torch.bfloat16, device="cuda")
    hm.gemm(1, x, packed, n, k, out=y)
    torch.cuda.synchronize()
    assert hm.device_error() & 1
    assert (y == 7.0).all()


def test_full_size_layers_sampled(hm):
    """The benchmark's three layers at M = 1 and 16 from the device generators, checked on 256
    sampled outputs each (the oracle quantizes host copies of the sampled weight rows)."""
    from oracle import quant as oq
    rng = np.random.default_rng(9)
    for n, k in ((4096, 4096), (14336, 4096), (4096, 14336)):
        d = hm.desc(1, n, k, True)
        w = synth.device_weights(n, k, seed=n + k)
        z = synth.device_zero_points(n, k // 128, seed=n + k + 1)
        q, s, _ = hm.quantize_weight(d, w, z)
        packed = hm.transform(d, q, s, z)
        for m in (1, 16):
            x = synth.device_activations(m, k, seed=m + n)
            y = hm.gemm(1, x, packed, n, k)
            torch.cuda.synchronize()
            ms = rng.integers(0, m, size=256)
            ns = rng.integers(0, n, size=256)
            wq, sq = oq.quant_int4(w[torch.from_numpy(ns).cuda()].cpu().numpy().astype(np.float64),
                                   zeros=z[torch.from_numpy(ns).cuda()].cpu().numpy())
            what = oq.dequant_int4(wq, sq, z[torch.from_numpy(ns).cuda()].cpu().numpy())
            ref = np.einsum("ik,ik->i", bf16_np(x)[ms], what)
            got = bf16_np(y.cpu()[torch.from_numpy(ms), torch.from_numpy(ns)])
            ok = og.tolerance_ok(got, ref)
            assert ok.all(), f"{n}x{k} M={m}: {int((~ok).sum())} of 256 outside tolerance"
        del w, q, s, packed
    assert hm.device_error() == 0
