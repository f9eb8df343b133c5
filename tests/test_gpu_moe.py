"""GPU parity of the grouped MoE GEMM (W4A16 INT4 and MXFP4-W4A16) against the oracle's
per-expert product over expert-sorted rows."""
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


def moe_case(hm, fmt, counts, n, k, has_zero=False, seed=0, gain=1.0):
    e = len(counts)
    offsets = np.zeros(e + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    rows = int(offsets[-1])
    qws, packs = [], []
    for i in range(e):
        z = synth.zero_points(n, k // 128, seed=seed + 100 + i) if has_zero else None
        qw = QuantWeight(fmt, synth.weights(n, k, seed=seed + i) * np.float32(gain), z)
        qws.append(qw)
        packs.append(qw.transform(hm)[1])
    ptrs = torch.tensor([p.data_ptr() for p in packs], dtype=torch.int64, device="cuda")
    x = synth.activations(rows, k, seed=seed + 999)
    full, y = canary_out(rows, n)
    hm.moe_gemm(fmt, x.cuda(), torch.from_numpy(offsets).cuda(), ptrs, n, k, out=y)
    torch.cuda.synchronize()
    yref = og.moe_gemm(bf16_np(x), offsets, [q.what for q in qws])
    assert_close(y, yref, f"moe fmt={fmt} counts={counts}")
    check_canary(full, rows, f"moe fmt={fmt} counts={counts}")
    assert hm.device_error() == 0
    return y


@pytest.mark.parametrize("fmt", [1, 2])
def test_skewed_with_empty_experts(hm, fmt):
    moe_case(hm, fmt, [37, 0, 1, 200, 0, 5, 16, 0], 256, 512, has_zero=(fmt == 1))


def test_single_expert_equals_dense(hm):
    n, k, m = 384, 1024, 70
    qw = QuantWeight(1, synth.weights(n, k, seed=1), synth.zero_points(n, k // 128, seed=2))
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=3).cuda()
    ptrs = torch.tensor([packed.data_ptr()], dtype=torch.int64, device="cuda")
    y_moe = hm.moe_gemm(1, x, torch.tensor([0, m], dtype=torch.int32, device="cuda"), ptrs, n, k)
    y_dense = hm.gemm(1, x, packed, n, k)
    torch.cuda.synchronize()
    assert_close(y_moe, og.gemm(bf16_np(x), qw.what), "single expert")
    assert_close(y_dense, og.gemm(bf16_np(x), qw.what), "dense")


def test_zipf_routing_small(hm):
    tok, exp, offsets = synth.moe_routing(tokens=64, experts=16, topk=4, seed=0)
    counts = np.diff(offsets).tolist()
    moe_case(hm, 1, counts, 256, 256, has_zero=True, seed=3)


def test_bad_offsets_set_device_error(hm):
    n, k = 128, 128
    qw = QuantWeight(1, synth.weights(n, k, seed=1))
    _, packed = qw.transform(hm)
    ptrs = torch.tensor([packed.data_ptr()] * 2, dtype=torch.int64, device="cuda")
    x = synth.activations(8, k, seed=2).cuda()
    offs = torch.tensor([0, 6, 3], dtype=torch.int32, device="cuda")   # decreasing
    hm.moe_gemm(1, x, offs, ptrs, n, k)
    assert hm.device_error() & 4


@pytest.mark.parametrize("fmt", [1, 2])
def test_offsets_past_rows_abort_before_any_store(hm, fmt):
    """Offsets that run past the rows (here 100 > 8) set the offsets error and stop the kernel
    before any tile is stored: the rows after Y keep their contents. INT4 runs the small-token
    kernel at this size, MXFP4 the general one."""
    n, k = 128, 256
    qw = QuantWeight(fmt, synth.weights(n, k, seed=1))
    _, packed = qw.transform(hm)
    ptrs = torch.tensor([packed.data_ptr()], dtype=torch.int64, device="cuda")
    x = synth.activations(8, k, seed=2).cuda()
    y = torch.full((128, n), 7.0, dtype=torch.bfloat16, device="cuda")
    offs = torch.tensor([0, 100], dtype=torch.int32, device="cuda")
    hm.moe_gemm(fmt, x, offs, ptrs, n, k, out=y[:8])
    torch.cuda.synchronize()
    assert hm.device_error() & 4
    assert (y[8:] == 7.0).all()


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("small", ["0", "1"])
def test_small_tiles_both_kernels(hm, fmt, small, monkeypatch):
    """Token tiles of 16 and 32: INT4 runs the small-token kernel (the general kernel with
    HM_F16_SMALL=0), MXFP4 the general kernel (its restore is heavier than the small-token kernel's
    dequant warps keep up with: measured slower there)."""
    monkeypatch.setenv("HM_F16_SMALL", small)
    monkeypatch.setenv("HM_MOE_TILE_M", "16")
    moe_case(hm, fmt, [3, 0, 17, 40, 1, 0, 9], 256, 1024, has_zero=(fmt == 1), seed=11)
    monkeypatch.setenv("HM_MOE_TILE_M", "32")
    moe_case(hm, fmt, [3, 0, 17, 40, 1, 0, 9], 256, 1024, has_zero=False, seed=12)


@pytest.mark.parametrize("tile", ["16", "32"])
def test_small_tiles_mxfp4_large_scales(hm, tile, monkeypatch):
    """MXFP4 blocks with E8M0 exponents above 128 (fp32 restore) at token tiles of 16 and 32."""
    monkeypatch.setenv("HM_MOE_TILE_M", tile)
    moe_case(hm, 2, [5, 0, 12, 30], 256, 512, seed=31, gain=2.0 ** 14)


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("tile", ["64", "128", "256"])
def test_forced_token_tiles(hm, fmt, tile, monkeypatch):
    """Every token tile of the grouped path, including the 256-row tile with restored weights in
    shared memory, on skewed counts with empty experts and experts larger than the tile."""
    monkeypatch.setenv("HM_MOE_TILE_M", tile)
    moe_case(hm, fmt, [300, 0, 1, 17, 0, 129, 256, 3], 256, 512, has_zero=(fmt == 1), seed=21)
