"""GPU parity of the MXINT4-W4A16 path (signed 4-bit integers with an E8M0 scale per 32 along
K, restored q * 2^(e-127)) through the C ABI against the fp64 oracle: the quantizer and the
transform byte for byte, the dequant hook bit for bit, the decode kernel (M <= 32) on the
hand-off shapes, the tcgen05 kernel on every token tile with and without stream-K, extreme
scales, and the grouped MoE product. GEMM tolerance |Y - Yref| <= 1e-2*|Yref| + 1e-2*rms(Yref)."""
import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import gemm as og
from oracle import quant as oq

from .gpu_util import QuantWeight, assert_close, bf16_np, canary_out, check_canary, pack_nibbles

pytestmark = pytest.mark.gpu

FMT = 5
_cache = {}


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


def weight(hm, n, k, seed, gain=1.0):
    key = (n, k, seed, gain)
    if key not in _cache:
        qw = QuantWeight(FMT, synth.weights(n, k, seed=seed) * np.float32(gain))
        _cache[key] = (qw, qw.transform(hm)[1])
    return _cache[key]


def gemm_case(hm, m, n, k, seed=0, gain=1.0, what=""):
    qw, packed = weight(hm, n, k, seed, gain)
    x = synth.activations(m, k, seed=seed + 2)
    full, y = canary_out(m, n)
    hm.gemm(FMT, x.cuda(), packed, n, k, out=y)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"mxint4 m={m} n={n} k={k} {what}")
    check_canary(full, m, f"mxint4 m={m} n={n} k={k}")
    assert hm.device_error() == 0


@pytest.mark.parametrize("n,k", [(256, 512), (100, 128), (130, 1024)])
def test_quantize_and_transform(hm, n, k):
    w = synth.weights(n, k, seed=13)
    w[0, :32] = 0.0                                   # an all-zero block: e = 0, q = 0
    w[1, 5] = 0.5                                     # a block with a large outlier
    w[2, 32:64] = np.float32(1.875) * np.sign(w[2, 32:64])   # ties at +-7.5 X
    q, e = oq.quant_mxint4(w)
    d = hm.desc(FMT, n, k)
    qg, sg, _ = hm.quantize_weight(d, torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(sg.cpu().numpy(), e.astype(np.uint8))
    np.testing.assert_array_equal(qg.cpu().numpy(), pack_nibbles(q))
    qw = QuantWeight(FMT, w)
    _, packed = qw.transform(hm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(packed.cpu().numpy(), qw.packed_ref)


@pytest.mark.parametrize("log2_gain", [0, -100, -122, 120])
def test_dequant_hook_bit_exact(hm, log2_gain):
    """Restored bf16 weights equal q * 2^(e-127) exactly, including e = 0 (the subnormal scale
    2^-127) and large exponents."""
    n, k = 130, 256
    w = synth.weights(n, k, seed=21) * np.float32(2.0 ** log2_gain)
    qw = QuantWeight(FMT, w)
    d, packed = qw.transform(hm)
    if log2_gain == -122:                             # every block at e = 0, codes up to +-3
        assert (qw.s == 0).all() and (qw.q != 0).any()
    wd = hm.dequant(d, packed)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_np(wd), qw.what)


# (n, k): tiles cut into many K ranges (global hand-off) | ragged N, one block | clusters of 2
# (the hand-offs are shared with the other W4A16 formats, tested on more shapes there)
@pytest.mark.parametrize("n,k", [(640, 3072), (200, 128), (8192, 1024)])
@pytest.mark.parametrize("m", [1, 7, 16, 32])
def test_decode_kernel(hm, m, n, k):
    p = hm.plan(FMT, m, n, k, torch.cuda.get_device_properties(0).multi_processor_count)
    assert p["kernel"] == 1 and p["tile_m"] >= m
    gemm_case(hm, m, n, k, seed=400)


@pytest.mark.parametrize("m", [33, 64, 100, 256, 300])
def test_tcgen05_m_sweep(hm, m):
    gemm_case(hm, m, 384, 1024, seed=410)


@pytest.mark.parametrize("tile_m", ["16", "32", "64", "128", "192", "256"])
@pytest.mark.parametrize("stream_k", ["0", "1"])
def test_tcgen05_forced_tiles(hm, monkeypatch, tile_m, stream_k):
    monkeypatch.setenv("HM_GEMV", "0")
    monkeypatch.setenv("HM_TILE_M", tile_m)
    monkeypatch.setenv("HM_STREAM_K", stream_k)
    gemm_case(hm, 70, 512, 2048, seed=420, what=f"tile {tile_m} sk {stream_k}")


@pytest.mark.parametrize("log2_gain", [-100, 14, 120])
@pytest.mark.parametrize("m", [5, 70])
def test_extreme_scales(hm, m, log2_gain):
    gemm_case(hm, m, 256, 512, seed=430, gain=2.0 ** log2_gain, what=f"gain 2^{log2_gain}")


@pytest.mark.parametrize("tile", ["16", "32", "64", "128", "256"])
def test_moe(hm, monkeypatch, tile):
    monkeypatch.setenv("HM_MOE_TILE_M", tile)
    counts = [37, 0, 1, 200, 0, 5, 16, 0]
    n, k = 256, 512
    offsets = np.zeros(len(counts) + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    ws = [weight(hm, n, k, seed=440 + i) for i in range(len(counts))]
    ptrs = torch.tensor([p.data_ptr() for _, p in ws], dtype=torch.int64, device="cuda")
    x = synth.activations(int(offsets[-1]), k, seed=449)
    y = hm.moe_gemm(FMT, x.cuda(), torch.from_numpy(offsets).cuda(), ptrs, n, k)
    torch.cuda.synchronize()
    assert_close(y, og.moe_gemm(bf16_np(x), offsets, [qw.what for qw, _ in ws]), f"moe tile {tile}")
    assert hm.device_error() == 0
