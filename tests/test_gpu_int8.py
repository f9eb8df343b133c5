"""GPU parity of the INT8 weight format with bf16 activations (HM_W8A16_INT8), through the C ABI:
the quantizer and transform byte for byte against the oracle, the dequant hook bit for bit, the GEMM
on the decode kernel (M <= 32) and on every tcgen05 token tile (16 .. 192, with and without a K
split) within the GEMM tolerance, symmetric and with u8 zero-points, and the grouped MoE."""
import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import formats as of
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


def u8_zeros(n, groups, seed):
    return np.random.default_rng(seed).integers(0, 256, size=(n, groups), dtype=np.uint8)


@pytest.mark.parametrize("has_zero", [False, True])
@pytest.mark.parametrize("n,k", [(200, 512), (130, 1024)])
def test_quantizer_transform_dequant_exact(hm, has_zero, n, k):
    w = synth.weights(n, k, seed=51)
    w[4, :128] = 0.0                                   # an all-zero group
    w[5, 7] = 0.9                                      # an outlier
    z = u8_zeros(n, k // 128, 52) if has_zero else None
    q, s = oq.quant_int8(w, zeros=z)
    d = hm.desc(7, n, k, has_zero)
    qg, sg, _ = hm.quantize_weight(d, torch.from_numpy(w).cuda(), None if z is None else torch.from_numpy(z).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(qg.cpu().numpy(), (q & 0xFF).astype(np.uint8))
    np.testing.assert_array_equal(sg.view(torch.uint16).cpu().numpy(), of.bf16_bits(s))
    qw = QuantWeight(7, w, z)
    _, packed = qw.transform(hm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(packed.cpu().numpy(), qw.packed_ref)
    wd = hm.dequant(qw.desc(hm), packed)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_np(wd), qw.what)
    assert hm.device_error() == 0


@pytest.mark.parametrize("has_zero", [False, True])
@pytest.mark.parametrize("m", [1, 5, 8, 16, 17, 32, 33, 64, 130, 300])
def test_gemm_matches_oracle(hm, has_zero, m):
    n, k = 384, 1024
    w = synth.weights(n, k, seed=53)
    z = u8_zeros(n, k // 128, 54) if has_zero else None
    qw = QuantWeight(7, w, z)
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=55 + m)
    full, y = canary_out(m, n)
    hm.gemm(7, x.cuda(), packed, n, k, out=y)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"int8 M={m}")
    check_canary(full, m, "int8")
    assert hm.device_error() == 0


@pytest.mark.parametrize("tile", ["16", "32", "64", "128", "192"])
@pytest.mark.parametrize("stream_k", ["0", "1"])
def test_every_tcgen05_tile(hm, tile, stream_k, monkeypatch):
    monkeypatch.setenv("HM_GEMV", "0")
    monkeypatch.setenv("HM_TILE_M", tile)
    monkeypatch.setenv("HM_STREAM_K", stream_k)
    n, k, m = 256, 1024, 210
    qw = QuantWeight(7, synth.weights(n, k, seed=56), u8_zeros(n, k // 128, 57))
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=58)
    y = hm.gemm(7, x.cuda(), packed, n, k)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"int8 tile {tile} stream-K {stream_k}")
    assert hm.device_error() == 0


def test_split_decode_shapes(hm):
    """Decode-kernel splits of one tile along K (thread-block cluster) and across tiles."""
    for n, k, m in ((4096, 4096, 1), (640, 8192, 8), (1024, 2048, 32)):
        qw = QuantWeight(7, synth.weights(n, k, seed=59))
        _, packed = qw.transform(hm)
        x = synth.activations(m, k, seed=60)
        y = hm.gemm(7, x.cuda(), packed, n, k)
        torch.cuda.synchronize()
        assert_close(y, og.gemm(bf16_np(x), qw.what), f"int8 {n}x{k} M={m}")
    assert hm.device_error() == 0


@pytest.mark.parametrize("tile", ["16", "64", "128"])
def test_grouped_moe(hm, tile, monkeypatch):
    monkeypatch.setenv("HM_MOE_TILE_M", tile)
    counts = [37, 0, 1, 200, 0, 5, 16, 0]
    n, k = 256, 512
    offsets = np.zeros(len(counts) + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    rows = int(offsets[-1])
    qws = [QuantWeight(7, synth.weights(n, k, seed=70 + e), u8_zeros(n, k // 128, 80 + e)) for e in range(len(counts))]
    packs = [q.transform(hm)[1] for q in qws]
    ptrs = torch.tensor([p.data_ptr() for p in packs], dtype=torch.int64, device="cuda")
    x = synth.activations(rows, k, seed=71)
    y = hm.moe_gemm(7, x.cuda(), torch.from_numpy(offsets).cuda(), ptrs, n, k)
    torch.cuda.synchronize()
    assert_close(y, og.moe_gemm(bf16_np(x), offsets, [q.what for q in qws]), f"int8 moe tile {tile}")
    assert hm.device_error() == 0
