"""GPU parity of the activation quantizers (bit-exact against the oracle)."""
import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
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
