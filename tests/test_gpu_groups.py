"""GPU parity of the INT4 group sizes and zero-point conventions (the weights "from different
quantization tools" brought into one standard format, aihaber.org, section "Mimari"):

* HM_W4A16_INT4 with groups of 256, 512 and one scale per row (per channel), which the transform
  spreads over the 128-K units;
* HM_W4A16_INT4_G32 with groups of 32 and 64 (a bf16 scale and u4 zero-point per 32-K chunk);
* zero-points handed over in the GPTQ-style convention (stored z - 1 mod 16).

The quantizer and transform are compared byte for byte with the oracle, the dequant hook bit for bit,
the GEMM (decode kernel, every tcgen05 token tile, grouped MoE) within the GEMM tolerance."""
import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import formats as of
from oracle import gemm as og
from oracle import quant as oq

from .gpu_util import QuantWeight, assert_close, bf16_np, pack_nibbles

pytestmark = pytest.mark.gpu

CASES = [(1, 256, True), (1, 512, False), (1, -1, True), (6, 32, True), (6, 32, False), (6, 64, True)]


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


def _grp(fmt, group, k):
    return k if group == -1 else group


@pytest.mark.parametrize("fmt,group,has_zero", CASES)
def test_quantizer_and_transform_byte_exact(hm, fmt, group, has_zero):
    n, k = 200, 1024
    g = _grp(fmt, group, k)
    w = synth.weights(n, k, seed=21)
    w[3, :g] = 0.0                                    # an all-zero group
    z = synth.zero_points(n, k // g, seed=22) if has_zero else None
    q, s = oq.quant_int4(w, zeros=z, group=g)
    d = hm.desc(fmt, n, k, has_zero, group=group)
    qg, sg, _ = hm.quantize_weight(d, torch.from_numpy(w).cuda(), None if z is None else torch.from_numpy(z).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(qg.cpu().numpy(), pack_nibbles(q))
    np.testing.assert_array_equal(sg.view(torch.uint16).cpu().numpy(), of.bf16_bits(s))
    qw = QuantWeight(fmt, w, z, group=group)
    _, packed = qw.transform(hm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(packed.cpu().numpy(), qw.packed_ref)
    wd = hm.dequant(qw.desc(hm), packed)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_np(wd), qw.what)
    assert hm.device_error() == 0


@pytest.mark.parametrize("fmt,group", [(1, 256), (6, 32), (6, 64)])
def test_gptq_zero_convention_packs_the_same(hm, fmt, group):
    n, k = 130, 512
    w = synth.weights(n, k, seed=23)
    z = synth.zero_points(n, k // group, seed=24)
    z[0, 0] = 0                                       # the value whose stored form wraps to 15
    qw = QuantWeight(fmt, w, z, group=group)
    q, s, _ = qw.device_inputs()
    stored = torch.from_numpy(oq.gptq_stored_zero(z).astype(np.uint8)).cuda()
    packed = hm.transform(qw.desc(hm, zero_convention=hm.ZP_GPTQ), q, s, stored)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(packed.cpu().numpy(), qw.packed_ref)


@pytest.mark.parametrize("fmt,group,has_zero", CASES)
@pytest.mark.parametrize("m", [1, 8, 16, 32, 64, 200])
def test_gemm_matches_oracle(hm, fmt, group, has_zero, m):
    n, k = 384, 1024
    g = _grp(fmt, group, k)
    w = synth.weights(n, k, seed=25)
    z = synth.zero_points(n, k // g, seed=26) if has_zero else None
    qw = QuantWeight(fmt, w, z, group=group)
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=27 + m)
    y = hm.gemm(fmt, x.cuda(), packed, n, k)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"fmt={fmt} group={group} M={m}")
    assert hm.device_error() == 0


@pytest.mark.parametrize("tile", ["16", "32", "64", "128", "192", "256"])
@pytest.mark.parametrize("stream_k", ["0", "1"])
def test_g32_every_tcgen05_tile(hm, tile, stream_k, monkeypatch):
    monkeypatch.setenv("HM_GEMV", "0")
    monkeypatch.setenv("HM_TILE_M", tile)
    monkeypatch.setenv("HM_STREAM_K", stream_k)
    n, k, m = 256, 1024, 150
    qw = QuantWeight(6, synth.weights(n, k, seed=28), synth.zero_points(n, k // 32, seed=29), group=32)
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=30)
    y = hm.gemm(6, x.cuda(), packed, n, k)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), f"tile {tile} stream-K {stream_k}")
    assert hm.device_error() == 0


@pytest.mark.parametrize("group", [32, 64])
def test_g32_grouped_moe(hm, group):
    counts = [37, 0, 1, 200, 0, 5, 16, 0]
    n, k = 256, 512
    offsets = np.zeros(len(counts) + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    rows = int(offsets[-1])
    qws = [QuantWeight(6, synth.weights(n, k, seed=40 + e), synth.zero_points(n, k // group, seed=60 + e), group=group)
           for e in range(len(counts))]
    packs = [q.transform(hm)[1] for q in qws]
    ptrs = torch.tensor([p.data_ptr() for p in packs], dtype=torch.int64, device="cuda")
    x = synth.activations(rows, k, seed=41)
    y = hm.moe_gemm(6, x.cuda(), torch.from_numpy(offsets).cuda(), ptrs, n, k)
    torch.cuda.synchronize()
    assert_close(y, og.moe_gemm(bf16_np(x), offsets, [q.what for q in qws]), f"g32 moe group {group}")
    assert hm.device_error() == 0
