"""GPU parity of the activation quantizers (bit-exact against the oracle) and of the MoE expert
activation SiLU(gate) * up (bf16 output within one bf16 step of the oracle's rounding of the exact
value, almost always equal)."""
import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import act as oa
from oracle import layout as ol
from oracle import quant as oq

from .gpu_util import pack_nibbles

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


@pytest.mark.parametrize("m,k", [(1, 7168), (5, 512), (130, 1024), (64, 16)])
def test_fp8_per_token(hm, m, k):
    x = synth.activations(m, k, seed=41, outlier_frac=0.01)
    if m > 2:
        x[2] = 0                          # a zero row
    xq, st = oq.quant_fp8_per_token(x.float().numpy())
    gq, gs = hm.quant_act_fp8(x.cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gs.cpu().numpy().astype(np.float64), st)
    np.testing.assert_array_equal(gq.cpu().numpy(), xq)


@pytest.mark.parametrize("m,k", [(1, 512), (16, 8192), (130, 1024), (128, 64)])
def test_nvfp4_act(hm, m, k):
    x = synth.activations(m, k, seed=42)
    codes, sb, g = oq.quant_nvfp4(x.float().numpy())
    body, atoms = ol.pack_act_nvfp4(codes, sb)
    gq, gs, gg = hm.quant_act_nvfp4(x.cuda())
    torch.cuda.synchronize()
    assert float(gg.item()) == g
    np.testing.assert_array_equal(gq.cpu().numpy(), body)
    np.testing.assert_array_equal(gs.cpu().numpy(), atoms)


def test_nvfp4_act_given_scale(hm):
    m, k = 40, 256
    x = synth.activations(m, k, seed=43)
    g = 0.01
    codes, sb, _ = oq.quant_nvfp4(x.float().numpy(), g=np.float32(g))
    gq, gs, gg = hm.quant_act_nvfp4(x.cuda(), g_in=torch.tensor([g], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert float(gg.item()) == np.float32(g)
    np.testing.assert_array_equal(gq.cpu().numpy(), pack_nibbles(codes))
    _, atoms = ol.pack_act_nvfp4(codes, sb)
    np.testing.assert_array_equal(gs.cpu().numpy(), atoms)


def test_nvfp4_act_all_zero(hm):
    """An all-zero X: the tensor scale is 1 by the reading taken, every block scale and code 0."""
    m, k = 3, 128
    x = torch.zeros((m, k), dtype=torch.bfloat16)
    codes, sb, g = oq.quant_nvfp4(x.float().numpy())
    assert g == 1.0 and not codes.any() and not sb.any()
    gq, gs, gg = hm.quant_act_nvfp4(x.cuda())
    torch.cuda.synchronize()
    assert float(gg.item()) == 1.0
    assert not gq.cpu().numpy().any()
    np.testing.assert_array_equal(gs.cpu().numpy(), ol.pack_act_nvfp4(codes, sb)[1])


def _bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("rows,inter", [(1, 8), (3, 2048), (130, 1024), (257, 56), (1024, 4096)])
def test_silu_mul(hm, rows, inter):
    """The kernel evaluates SiLU in fp32 (expf) and rounds the product once to bf16; the oracle
    rounds the exact fp64 value. They differ by at most one bf16 step (a near-tie of the fp32
    result), rarely."""
    gu = synth.activations(rows, 2 * inter, seed=50 + rows)
    gu[:, : inter // 2] *= 8.0                      # gates from about -40 to 40 (both asymptotes)
    if rows > 2:
        gu[1, :inter] = 0.0                          # zero gates give zero
        # gates out to +-100: exp(g) underflows fp32 below about -87 where SiLU is still a bf16 number
        gu[2, :inter] = torch.linspace(-100.0, 100.0, inter).to(torch.bfloat16)
    ref = oa.silu_mul(gu.float().numpy(), inter)
    got = hm.silu_mul(gu.cuda(), inter)
    torch.cuda.synchronize()
    g = got.float().cpu().numpy().astype(np.float64)
    diff = np.abs(g - ref)
    assert (diff <= _bf16_ulp(ref) + 1e-45).all(), f"max diff {diff.max()}"
    assert (diff == 0).mean() >= 0.99
    if rows > 2:
        assert (g[1] == 0).all()
    assert hm.device_error() == 0


def test_silu_mul_writes_only_its_rows(hm):
    """On a whole gate-up output the kernel writes exactly rows x inter values; a strided slice
    and a mis-shaped output are refused by the binding; zero rows is a no-op."""
    rows, inter = 64, 512
    gu = synth.activations(rows, 2 * inter, seed=77).cuda()
    out = torch.full((rows + 1, inter), 7.0, dtype=torch.bfloat16, device="cuda")
    hm.silu_mul(gu, inter, out=out[:rows])
    torch.cuda.synchronize()
    assert (out[rows] == 7.0).all()                  # the row after the output is untouched
    with pytest.raises(AssertionError):
        hm.silu_mul(gu[:, ::2], inter // 2)
    with pytest.raises(AssertionError):
        hm.silu_mul(gu, inter, out=out)
    empty = hm.silu_mul(gu[:0], inter)
    torch.cuda.synchronize()
    assert empty.shape == (0, inter)
