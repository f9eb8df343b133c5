"""The allocation-free W4A16 entry point (hm_gemm_w4a16_noalloc).

Some callers cannot allocate device memory: code running inside another engine's fixed
memory plan, or code that must not call cudaMalloc because it synchronises the device. For
them the library keeps the split-K scratch in an array of its own. This file checks, through
the C ABI, that two calls in a row give the same output as hm_gemm with a caller workspace
(within the GEMM tolerance), and that a problem too large for the built-in scratch is
rejected. It is collected last so that a failure here never hides another test's result.
"""
import ctypes

import pytest
import torch

from moe_hm_gemm_gb300 import synth

from .gpu_util import QuantWeight

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


def _close(a, b):
    from oracle import gemm as og
    ok = og.tolerance_ok(a.float().cpu().numpy(), b.float().cpu().numpy())
    return bool(ok.all()), int((~ok).sum())


@pytest.mark.parametrize("fmt,m,n,k", [(1, 1, 4096, 4096), (1, 16, 1024, 2048), (2, 8, 512, 1024),
                                       (1, 64, 384, 1024)])
def test_noalloc_matches_workspace_entry_twice(hm, fmt, m, n, k):
    has_zero = fmt == 1
    w = synth.weights(n, k, seed=5)
    z = synth.zero_points(n, k // 128, seed=6) if has_zero else None
    qw = QuantWeight(fmt, w, z)
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=7).cuda()
    y_ref = hm.gemm(fmt, x, packed, n, k)
    for _ in range(2):                       # two calls in a row share the library's scratch
        y = hm.gemm_noalloc(fmt, x, packed, n, k)
        torch.cuda.synchronize()
        ok, bad = _close(y, y_ref)
        assert ok, f"{bad} outputs differ beyond tolerance"
    assert hm.device_error() == 0


def test_noalloc_rejects_problems_beyond_its_scratch(hm):
    lib = hm.lib()
    P = ctypes.c_void_p
    x = torch.empty((4096, 4096), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((4096, 4096), dtype=torch.bfloat16, device="cuda")
    packed = torch.empty((hm.packed_size(hm.desc(1, 4096, 4096)),), dtype=torch.uint8, device="cuda")
    # M = 200 needs tile_m 128 with stream-K: far more than 8 MiB of partials
    status = lib.hm_gemm_w4a16_noalloc(1, P(x.data_ptr()), P(packed.data_ptr()), P(y.data_ptr()), 200, 4096, 4096,
                                       P(torch.cuda.current_stream().cuda_stream))
    assert status == 3                       # HM_ERR_WORKSPACE: nothing launched
    assert lib.hm_gemm_w4a16_noalloc(3, P(x.data_ptr()), P(packed.data_ptr()), P(y.data_ptr()), 4, 4096, 4096,
                                     None) == 1
