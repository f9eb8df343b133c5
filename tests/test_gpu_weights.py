"""GPU parity of the weight path through the C ABI: the RNE quantizer, the transform (byte
for byte against the oracle's layout) and the dequant hook (bitwise against the oracle's
restored weights). Integer / byte work is compared exactly."""
import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import formats as of
from oracle import layout as ol
from oracle import quant as oq

from .gpu_util import QuantWeight, pack_nibbles

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


SHAPES = [(256, 512), (200, 384), (130, 1024)]


@pytest.mark.parametrize("n,k", SHAPES)
@pytest.mark.parametrize("has_zero", [False, True])
def test_quantize_int4(hm, n, k, has_zero):
    w = synth.weights(n, k, seed=11)
    z = synth.zero_points(n, k // 128, seed=12) if has_zero else None
    q, s = oq.quant_int4(w, zeros=z)
    d = hm.desc(1, n, k, has_zero)
    qg, sg, _ = hm.quantize_weight(d, torch.from_numpy(w).cuda(), None if z is None else torch.from_numpy(z).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(qg.cpu().numpy(), pack_nibbles(q))
    np.testing.assert_array_equal(sg.view(torch.uint16).cpu().numpy(), of.bf16_bits(s))


@pytest.mark.parametrize("n,k", SHAPES)
def test_quantize_mxfp4(hm, n, k):
    w = synth.weights(n, k, seed=13)
    w[0, :32] = 0.0                      # an all-zero block
    w[1, 5] = 0.5                        # a block with a large outlier
    codes, e = oq.quant_mxfp4(w)
    qg, sg, _ = hm.quantize_weight(hm.desc(3, n, k), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(sg.cpu().numpy(), e.astype(np.uint8))
    np.testing.assert_array_equal(qg.cpu().numpy(), pack_nibbles(codes))


def test_quantize_nvfp4_tensor_scale_not_one(hm):
    """The hand-computed NVFP4 row of the oracle's tests (tensor amax 1, g = fp32(1/2688)), every
    value at a rounding boundary of one step of the recipe, quantized on the GPU: the codes and
    scales written out there by hand."""
    def f(h):
        return float(np.array([h], dtype=np.uint32).view(np.float32)[0])
    w = np.zeros((2, 64), dtype=np.float32)
    w[0, 0] = 1.0
    w[0, 16:21] = [f(0x3B76DB6D), f(0x392AAAAB), f(0x3A955555), f(0x3A000000), -f(0x3A955555)]
    w[0, 32:36] = [f(0x3B400001), f(0x39C92492), f(0x3A279E7B), -f(0x3A279E7B)]
    w[0, 48:50] = [f(0x3B2DB6DB), -f(0x3B2DB6DB)]
    qg, sg, gg = hm.quantize_weight(hm.desc(4, 2, 64), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert gg.cpu().view(torch.int32).item() == 0x39C30C31
    expect = np.zeros((2, 64), dtype=np.int64)
    expect[0, 0] = 7
    expect[0, 16:21] = [7, 0, 3, 2, 11]
    expect[0, 32:36] = [7, 1, 2, 10]
    expect[0, 48:50] = [7, 15]
    np.testing.assert_array_equal(qg.cpu().numpy(), pack_nibbles(expect))
    np.testing.assert_array_equal(sg.cpu().numpy()[0], [0x7E, 0x3E, 0x3B, 0x39])
    assert not sg.cpu().numpy()[1].any()        # an all-zero row: sb = 0, codes 0


@pytest.mark.parametrize("n,k", [(256, 512), (100, 64), (130, 1024)])
def test_quantize_nvfp4(hm, n, k):
    w = synth.weights(n, k, seed=14)
    w[2, 16:32] = 0.0
    codes, sb, g = oq.quant_nvfp4(w)
    qg, sg, gg = hm.quantize_weight(hm.desc(4, n, k), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert float(gg.item()) == g
    np.testing.assert_array_equal(sg.cpu().numpy(), sb)
    np.testing.assert_array_equal(qg.cpu().numpy(), pack_nibbles(codes))


CASES = [(1, False), (1, True), (2, False), (3, False), (4, False)]


@pytest.mark.parametrize("fmt,has_zero", CASES)
@pytest.mark.parametrize("n,k", SHAPES)
def test_transform_bytes_and_dequant(hm, fmt, has_zero, n, k):
    w = synth.weights(n, k, seed=21)
    z = synth.zero_points(n, k // 128, seed=22) if has_zero else None
    qw = QuantWeight(fmt, w, z)
    d, packed = qw.transform(hm)
    torch.cuda.synchronize()
    got = packed.cpu().numpy()
    assert got.size == qw.packed_ref.size
    mism = np.nonzero(got != qw.packed_ref)[0]
    assert mism.size == 0, f"{mism.size} bytes differ, first at {mism[:8]}"
    wd = hm.dequant(d, packed)
    torch.cuda.synchronize()
    want = qw.what if fmt != 4 else oq.dequant_nvfp4(qw.q, qw.s, 1.0)   # NVFP4 hook omits gW
    want_bits = of.bf16_bits(of.bf16r(want))
    np.testing.assert_array_equal(wd.view(torch.uint16).cpu().numpy(), want_bits)


def test_transform_of_gpu_quantized_weights(hm):
    """Quantize on the GPU, transform, compare with the oracle's packed buffer (full chain)."""
    n, k = 384, 1024
    w = synth.weights(n, k, seed=31)
    z = synth.zero_points(n, k // 128, seed=32)
    d = hm.desc(1, n, k, True)
    q, s, _ = hm.quantize_weight(d, torch.from_numpy(w).cuda(), torch.from_numpy(z).cuda())
    packed = hm.transform(d, q, s, torch.from_numpy(z).cuda())
    torch.cuda.synchronize()
    ref = QuantWeight(ol.FMT_W4A16_INT4, w, z).packed_ref
    np.testing.assert_array_equal(packed.cpu().numpy(), ref)
