"""GPU parity of the W4A16 tcgen05 kernel run by CTA pairs (clusters of two CTAs sharing each
MMA: 256 weight rows per tile, each CTA holding half of the tile's activations), through the C
ABI, against the fp64 oracle with the tolerance |Y - Yref| <= 1e-2*|Yref| + 1e-2*rms(Yref) per
element; and agreement with the single-CTA kernel on the same inputs.

The pair path is taken for dense W4A16-family calls with 128- or 256-token tiles, whole tiles
per CTA and N a multiple of 256; HM_PAIR selects it (1) or keeps it off (0)."""
import os

import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import gemm as og
from oracle import layout as ol

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


def prepare(hm, fmt, n, k, has_zero, seed):
    w = synth.weights(n, k, seed=seed)
    g = 32 if fmt == ol.FMT_W4A16_INT4_G32 else 128      # zero-point (and scale) group along K
    z = None
    if has_zero and fmt == ol.FMT_W8A16_INT8:             # u8 zero-points
        z = np.random.default_rng(seed + 1).integers(0, 256, size=(n, k // g), dtype=np.uint8)
    elif has_zero:
        z = synth.zero_points(n, k // g, seed=seed + 1)
    qw = QuantWeight(fmt, w, z, group=32) if fmt == ol.FMT_W4A16_INT4_G32 else QuantWeight(fmt, w, z)
    _, packed = qw.transform(hm)
    return qw, packed


def run(hm, fmt, x, packed, n, k):
    m = x.shape[0]
    full, y = canary_out(m, n)
    hm.gemm(fmt, x, packed, n, k, out=y)
    torch.cuda.synchronize()
    check_canary(full, m, f"fmt={fmt} m={m} n={n} k={k}")
    assert hm.device_error() == 0
    return y


def assert_same_sums(y, y1, what):
    """The pair and single-CTA kernels add the same products in the same K order; at most a last-bit
    difference (one bf16 ulp) is accepted in case the tensor core groups a pair's sums differently."""
    if torch.equal(y, y1):
        return
    a, b = y.float(), y1.float()
    ulp = torch.maximum(a.abs(), b.abs()) * 2.0 ** -7
    assert bool(((a - b).abs() <= ulp).all()), f"{what}: pair and single-CTA results differ beyond one ulp"


def plan_of(hm, fmt, m, n, k):
    return hm.plan(fmt, m, n, k, torch.cuda.get_device_properties(0).multi_processor_count)


CASES = [
    # (fmt, tile_m, m, n, k, zero-points)
    (ol.FMT_W4A16_INT4, 128, 300, 512, 1024, True),      # ragged last token tile, two pair tiles
    (ol.FMT_W4A16_INT4, 256, 700, 768, 640, False),      # odd k-block count, three weight-row pairs
    (ol.FMT_W4A16_INT4, 128, 60, 256, 384, True),        # one tile, tokens only in the even CTA's half
    (ol.FMT_W4A16_INT4, 256, 129, 256, 256, True),       # odd CTA holds a single token
    (ol.FMT_W4A16_INT4_G32, 128, 200, 512, 512, True),
    (ol.FMT_W4A16_INT4_G32, 256, 300, 512, 512, False),
    (ol.FMT_W4A16_MXFP4, 128, 257, 512, 768, False),
    (ol.FMT_W4A16_MXFP4, 256, 513, 256, 512, False),
    (ol.FMT_W4A16_MXINT4, 256, 400, 512, 1024, False),
    (ol.FMT_W8A16_INT8, 128, 190, 512, 512, True),
]


@pytest.mark.parametrize("fmt,tile_m,m,n,k,zp", CASES)
def test_pair_parity(hm, env, fmt, tile_m, m, n, k, zp):
    env["HM_TILE_M"] = str(tile_m)
    env["HM_STREAM_K"] = "0"
    env["HM_PAIR"] = "1"
    p = plan_of(hm, fmt, m, n, k)
    assert p["tile_n"] == 256 and p["kernel"] == 0 and p["tile_m"] == tile_m, p
    qw, packed = prepare(hm, fmt, n, k, zp, seed=m + n)
    x = synth.activations(m, k, seed=m + 3)
    xd = x.cuda()
    y = run(hm, fmt, xd, packed, n, k)
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"pair fmt={fmt} tile={tile_m} m={m} n={n} k={k}")
    env["HM_PAIR"] = "0"
    assert plan_of(hm, fmt, m, n, k)["tile_n"] == 128
    y1 = run(hm, fmt, xd, packed, n, k)
    assert_same_sums(y, y1, f"fmt={fmt} tile={tile_m} m={m}")


def test_pair_not_taken_for_odd_weight_tiles(hm, env):
    """N = 640 (five 128-row tiles) cannot be cut into pairs: the single-CTA kernel runs."""
    env["HM_TILE_M"] = "128"
    env["HM_PAIR"] = "1"
    fmt, m, n, k = ol.FMT_W4A16_INT4, 300, 640, 512
    assert plan_of(hm, fmt, m, n, k)["tile_n"] == 128
    qw, packed = prepare(hm, fmt, n, k, True, seed=4)
    x = synth.activations(m, k, seed=5)
    y = run(hm, fmt, x.cuda(), packed, n, k)
    assert_close(y, og.gemm(bf16_np(x), qw.what), "N=640 with HM_PAIR=1")


def test_pair_deterministic_and_repeated(hm, env):
    """Back-to-back calls (the second starting while the first drains) give identical results."""
    env["HM_TILE_M"] = "256"
    env["HM_STREAM_K"] = "0"
    env["HM_PAIR"] = "1"
    fmt, m, n, k = ol.FMT_W4A16_INT4, 1024, 1024, 1024
    qw, packed = prepare(hm, fmt, n, k, True, seed=11)
    x = synth.activations(m, k, seed=12).cuda()
    ys = []
    for _ in range(3):
        y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        hm.gemm(fmt, x, packed, n, k, out=y)
        ys.append(y)
    torch.cuda.synchronize()
    assert hm.device_error() == 0
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])


@pytest.mark.parametrize("tile_m", [128, 256])
def test_pair_full_size_sampled(hm, env, tile_m):
    """The benchmark's 4096 x 4096 layer at M = 4096 (16 or 32 token tiles, 256 pair tiles over
    the device's pairs): sampled rows against the oracle, all of Y against the single-CTA kernel."""
    env["HM_TILE_M"] = str(tile_m)
    env["HM_STREAM_K"] = "0"
    env["HM_PAIR"] = "1"
    fmt, m, n, k = ol.FMT_W4A16_INT4, 4096, 4096, 4096
    qw, packed = prepare(hm, fmt, n, k, True, seed=21)
    x = synth.activations(m, k, seed=22)
    xd = x.cuda()
    y = run(hm, fmt, xd, packed, n, k)
    rows = np.random.default_rng(23).choice(m, 24, replace=False)
    xs = bf16_np(x)[rows]
    assert_close(y[torch.from_numpy(rows).cuda()], og.gemm(xs, qw.what), f"pair full size tile={tile_m}")
    env["HM_PAIR"] = "0"
    y1 = run(hm, fmt, xd, packed, n, k)
    assert_same_sums(y, y1, f"full size tile={tile_m}")
