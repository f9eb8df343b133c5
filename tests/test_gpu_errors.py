"""Device-side failure detection without faulting the GPU: a packed header that does not
match the call, and a pipeline wait that runs out (a barrier nothing completes, bounded to
a few milliseconds). Both set the device error word and return; the context stays usable."""
import pytest
import torch

from moe_hm_gemm_gb300 import synth

from .gpu_util import QuantWeight, assert_close, bf16_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


def test_wait_timeout_sets_error_and_context_survives(hm):
    assert hm.device_error() == 0
    hm.debug_wait_timeout(5_000_000)           # 5 ms
    assert hm.device_error() == 2
    assert hm.device_error() == 0              # read clears
    # the context still works
    from oracle import gemm as og
    qw = QuantWeight(1, synth.weights(128, 256, seed=1))
    _, packed = qw.transform(hm)
    x = synth.activations(4, 256, seed=2)
    y = hm.gemm(1, x.cuda(), packed, 128, 256)
    torch.cuda.synchronize()
    assert_close(y, og.gemm(bf16_np(x), qw.what), "after timeout")


def test_header_mismatch_sets_error(hm):
    qw = QuantWeight(1, synth.weights(256, 256, seed=1))
    _, packed = qw.transform(hm)
    x = synth.activations(4, 512, seed=2).cuda()
    hm.gemm(1, x, packed, 256, 512)            # K differs from the packed weight's
    assert hm.device_error() & 1
    hm.gemm(2, x[:, :256].contiguous(), packed, 256, 256)   # format differs
    assert hm.device_error() & 1
