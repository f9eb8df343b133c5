"""GPU parity of the grouped GEMM with the experts' packed weights at a fixed stride
(hm_moe_gemm_strided): the block-scaled W4A8-MXFP4 and W4A4-NVFP4 grouped MoE (activations
quantized inside the call, or, for W4A8, pre-quantized by the caller) and the W4A16 formats through
the same entry, against the oracle's per-expert product over expert-sorted rows; empty experts,
Zipf routing, every token tile, malformed offsets and a mismatched expert header."""
import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import gemm as og
from oracle import quant as oq
from oracle.formats import decode_e4m3

from .gpu_util import QuantWeight, assert_close, bf16_np, canary_out, check_canary

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


def strided_weights(hm, fmt, e, n, k, seed, has_zero=False):
    """E experts quantized by the oracle, transformed into one strided buffer."""
    qws = []
    d0 = hm.desc(fmt, n, k, has_zero)
    buf = hm.alloc_moe_packed(d0, e)
    for i in range(e):
        z = synth.zero_points(n, k // 128, seed=seed + 500 + i) if has_zero else None
        qw = QuantWeight(fmt, synth.weights(n, k, seed=seed + i), z)
        d = hm.desc(fmt, n, k, has_zero, qw.g)
        q, s, zz = qw.device_inputs()
        hm.transform(d, q, s, zz, out=hm.moe_expert_view(buf, d0, i))
        qws.append(qw)
    return buf, hm.moe_stride(d0), qws


def xhat_of(fmt, x):
    """The oracle's view of the activations the GEMM multiplies (quantized for A8 / A4)."""
    xv = bf16_np(x)
    if fmt == 3:
        xq, st = oq.quant_fp8_per_token(xv)
        return decode_e4m3(xq) * st[:, None]
    if fmt == 4:
        gx = oq.nvfp4_global_scale(xv)
        xc, xsb, _ = oq.quant_nvfp4(xv, g=gx)
        return oq.dequant_nvfp4(xc, xsb, gx)
    return xv


def strided_case(hm, fmt, counts, n, k, seed=0, has_zero=False, prequant=False):
    e = len(counts)
    offsets = np.zeros(e + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    rows = int(offsets[-1])
    buf, stride, qws = strided_weights(hm, fmt, e, n, k, seed, has_zero)
    x = synth.activations(rows, k, seed=seed + 999, outlier_frac=0.01 if fmt == 3 else 0.0)
    full, y = canary_out(rows, n)
    offs = torch.from_numpy(offsets).cuda()
    if prequant:
        xq, st = hm.quant_act_fp8(x.cuda())
        hm.moe_gemm_strided(fmt, xq, offs, buf, e, stride, n, k, x_scale=st, out=y)
    else:
        hm.moe_gemm_strided(fmt, x.cuda(), offs, buf, e, stride, n, k, out=y)
    torch.cuda.synchronize()
    yref = og.moe_gemm(xhat_of(fmt, x), offsets, [q.what for q in qws])
    assert_close(y, yref, f"strided moe fmt={fmt} counts={counts}")
    check_canary(full, rows, f"strided moe fmt={fmt}")
    assert hm.device_error() == 0
    return y


@pytest.mark.parametrize("fmt", [3, 4])
def test_block_scaled_skewed_with_empty_experts(hm, fmt):
    strided_case(hm, fmt, [37, 0, 1, 200, 0, 5, 16, 0], 256, 512, seed=1)


def test_w4a8_prequantized_activations(hm):
    strided_case(hm, 3, [3, 0, 40, 129, 1], 384, 1024, seed=2, prequant=True)


@pytest.mark.parametrize("fmt", [3, 4])
@pytest.mark.parametrize("tile", ["16", "32", "64", "128"])
def test_block_scaled_every_token_tile(hm, fmt, tile, monkeypatch):
    """Every token tile, on experts smaller and larger than the tile and empty ones; W4A4's scale
    atoms follow the expert token tiles of the chosen width."""
    monkeypatch.setenv("HM_MOE_TILE_M", tile)
    strided_case(hm, fmt, [300, 0, 1, 17, 0, 129, 64, 3], 256, 768, seed=3)


@pytest.mark.parametrize("fmt", [3, 4])
def test_block_scaled_zipf_routing(hm, fmt):
    _, _, offsets = synth.moe_routing(tokens=96, experts=32, topk=4, seed=1)
    strided_case(hm, fmt, np.diff(offsets).tolist(), 512, 1024, seed=4)


@pytest.mark.parametrize("fmt,has_zero", [(1, True), (1, False), (2, False), (5, False)])
def test_w4a16_formats_through_the_strided_entry(hm, fmt, has_zero):
    strided_case(hm, fmt, [20, 0, 3, 70, 1], 256, 512, seed=5, has_zero=has_zero)


def test_single_expert_equals_dense(hm):
    """One expert over all rows equals the dense GEMM of the same weight (W4A8, W4A4)."""
    for fmt in (3, 4):
        n, k, m = 256, 1024, 77
        buf, stride, qws = strided_weights(hm, fmt, 1, n, k, seed=6)
        x = synth.activations(m, k, seed=7).cuda()
        y_moe = hm.moe_gemm_strided(fmt, x, torch.tensor([0, m], dtype=torch.int32, device="cuda"), buf, 1, stride,
                                    n, k)
        torch.cuda.synchronize()
        assert_close(y_moe, og.gemm(xhat_of(fmt, x.cpu()), qws[0].what), f"single expert fmt={fmt}")
    assert hm.device_error() == 0


@pytest.mark.parametrize("fmt", [3, 4])
def test_bad_offsets_and_header_set_device_error(hm, fmt):
    n, k = 128, 256
    buf, stride, _ = strided_weights(hm, fmt, 2, n, k, seed=8)
    x = synth.activations(8, k, seed=9).cuda()
    y = torch.full((64, n), 7.0, dtype=torch.bfloat16, device="cuda")
    hm.moe_gemm_strided(fmt, x, torch.tensor([0, 6, 3], dtype=torch.int32, device="cuda"), buf, 2, stride, n, k,
                        out=y[:8])
    torch.cuda.synchronize()
    assert hm.device_error() & 4
    assert (y[8:] == 7.0).all()
    # the second expert's header made for another K
    buf2, stride2, _ = strided_weights(hm, fmt, 2, n, k, seed=10)
    other = hm.alloc_moe_packed(hm.desc(fmt, n, 2 * k), 1)
    qw = QuantWeight(fmt, synth.weights(n, 2 * k, seed=11))
    q, s, _ = qw.device_inputs()
    hm.transform(hm.desc(fmt, n, 2 * k, False, qw.g), q, s, None, out=other)
    buf2[stride2:stride2 + 256].copy_(other[:256])
    hm.moe_gemm_strided(fmt, x, torch.tensor([0, 4, 8], dtype=torch.int32, device="cuda"), buf2, 2, stride2, n, k)
    torch.cuda.synchronize()
    assert hm.device_error() & 1


@pytest.mark.parametrize("fmt", [3, 4])
def test_gate_up_full_size_sampled(hm, fmt):
    """E = 256 experts of the MoE gate-up layer (N = 4096, K = 7168), T = 4096 tokens with top-8
    Zipf(1.1) routing, checked on 256 sampled outputs: weights from the device generators, the oracle
    quantizing host copies of the sampled weight rows (row-local), activations quantized by the
    oracle from the same bf16 rows (W4A4: with the tensor scale of all rows)."""
    e, n, k, t = 256, 4096, 7168, 4096
    _, expert_of_row, offsets = synth.moe_routing(t, experts=e, topk=8, seed=0)
    rows = int(offsets[-1])
    rng = np.random.default_rng(5)
    rs = rng.integers(0, rows, size=256)
    ns = rng.integers(0, n, size=256)
    need = {}
    for i, r in enumerate(rs):
        need.setdefault(int(expert_of_row[r]), []).append(i)
    d0 = hm.desc(fmt, n, k)
    buf = hm.alloc_moe_packed(d0, e)
    w_rows = np.zeros((256, k))
    gws = np.zeros(256)
    for ei in range(e):
        w = synth.device_weights(n, k, seed=10000 + ei)
        q, s, g = hm.quantize_weight(d0, w)
        gw = float(g.item()) if fmt == 4 else 1.0
        hm.transform(hm.desc(fmt, n, k, False, gw), q, s, None, out=hm.moe_expert_view(buf, d0, ei))
        if need.get(ei) and fmt == 4:
            # the oracle's tensor scale from the whole matrix's amax (an exact max, taken on the device)
            g_ref = oq.nvfp4_global_scale(np.array([float(w.abs().max().item())]))
        for i in need.get(ei, []):
            w_rows[i] = w[int(ns[i])].cpu().numpy()
            gws[i] = g_ref if fmt == 4 else 1.0
        del w, q, s
    x = synth.device_activations(rows, k, seed=30000 + t, outlier_frac=0.01 if fmt == 3 else 0.0)
    y = hm.moe_gemm_strided(fmt, x, torch.from_numpy(offsets).cuda(), buf, e, hm.moe_stride(d0), n, k)
    torch.cuda.synchronize()
    assert hm.device_error() == 0
    if fmt == 3:
        what = oq.dequant_mxfp4(*oq.quant_mxfp4(w_rows))
        xq, st = oq.quant_fp8_per_token(bf16_np(x[torch.from_numpy(rs).cuda()]))
        xhat = decode_e4m3(xq) * st[:, None]
    else:
        what = np.zeros((256, k))
        for i in range(256):
            wc, wsb, _ = oq.quant_nvfp4(w_rows[i:i + 1], g=np.float32(gws[i]))
            what[i] = oq.dequant_nvfp4(wc, wsb, gws[i])[0]
        gx = oq.nvfp4_global_scale(bf16_np(x))
        xc, xsb, _ = oq.quant_nvfp4(bf16_np(x[torch.from_numpy(rs).cuda()]), g=gx)
        xhat = oq.dequant_nvfp4(xc, xsb, gx)
    ref = np.einsum("ik,ik->i", xhat, what)
    got = bf16_np(y[torch.from_numpy(rs).cuda(), torch.from_numpy(ns).cuda()])
    ok = og.tolerance_ok(got, ref)
    assert ok.all(), f"fmt={fmt}: {int((~ok).sum())} of 256 sampled outputs outside tolerance"
