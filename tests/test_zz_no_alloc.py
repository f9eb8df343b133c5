"""The allocation-free W4A16 entry point (hm_gemm_w4a16_noalloc).

Some callers cannot allocate device memory: code running inside another engine's fixed
memory plan, which hands it no workspace, or code that must not call cudaMalloc because that
call synchronises the device. For them the library keeps the split-K scratch in a fixed array
of its own. This file checks, through the C ABI, that two calls in a row give the output of
hm_gemm with a caller workspace and of the fp64 oracle (within the GEMM tolerance), for plans
that share tiles between CTAs (and so use the scratch) and plans that do not, and that a split
whose scratch would not fit the array is rejected with HM_ERR_WORKSPACE. It is collected last,
so that a failure here never hides another test's result.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import gemm as og

from .gpu_util import QuantWeight, assert_close

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 20 << 20        # the library's fixed array (stated in include/hm.h)


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


def _plan(hm, fmt, m, n, k):
    info = hm.PlanInfo()
    assert hm.lib().hm_plan(fmt, m, n, k, torch.cuda.get_device_properties(0).multi_processor_count,
                            ctypes.byref(info)) == 0
    return info


def _shares_tiles(info):
    return bool(info.stream_k) and (info.grid > info.tiles or info.tiles % info.grid != 0)


def _oracle_rows(qw, x, rows):
    xr = x[rows].float().cpu().numpy().astype(np.float64)
    return og.gemm(xr, qw.what)


# (fmt, M, N, K): decode-kernel splits, tcgen05 splits (the last one fills 16 MiB of the
# scratch), and plans that give every CTA whole tiles (M = 256 and 4096 on 4096x4096)
CASES = [(1, 1, 4096, 4096), (1, 16, 1024, 2048), (2, 8, 512, 1024), (1, 64, 384, 1024),
         (5, 64, 4096, 4096), (2, 128, 4096, 14336), (1, 256, 4096, 4096), (1, 4096, 4096, 4096)]


@pytest.mark.parametrize("fmt,m,n,k", CASES)
def test_noalloc_matches_workspace_entry_and_oracle_twice(hm, fmt, m, n, k):
    has_zero = fmt == 1
    w = synth.weights(n, k, seed=5)
    z = synth.zero_points(n, k // 128, seed=6) if has_zero else None
    qw = QuantWeight(fmt, w, z)
    _, packed = qw.transform(hm)
    x = synth.activations(m, k, seed=7).cuda()
    y_ws = hm.gemm(fmt, x, packed, n, k)         # the existing entry point, caller workspace
    rows = np.arange(m) if m <= 256 else np.random.default_rng(m).choice(m, 64, replace=False)
    yref = _oracle_rows(qw, x, rows)
    for call in range(2):                        # two calls in a row share the library's scratch
        y = hm.gemm_noalloc(fmt, x, packed, n, k)
        torch.cuda.synchronize()
        assert_close(y, y_ws.float().cpu().numpy().astype(np.float64), f"call {call} vs hm_gemm")
        assert_close(y[torch.from_numpy(rows).cuda()], yref, f"call {call} vs oracle")
    assert hm.device_error() == 0


def test_noalloc_plans_cover_both_kinds(hm):
    """The cases above include plans that share tiles (scratch used) and plans that do not."""
    kinds = {_shares_tiles(_plan(hm, *c)) for c in CASES}
    assert kinds == {True, False}


def test_noalloc_rejects_split_beyond_its_scratch(hm):
    lib = hm.lib()
    P = ctypes.c_void_p
    m, n, k = 256, 4096, 4096
    # force a split with 256-token tiles: 128 CTAs x 2 x 256 x 128 fp32 partials = 32 MiB
    old = {v: os.environ.get(v) for v in ("HM_TILE_M", "HM_STREAM_K")}
    os.environ["HM_TILE_M"], os.environ["HM_STREAM_K"] = "256", "1"
    try:
        info = _plan(hm, 2, m, n, k)
        assert _shares_tiles(info) and info.tile_m == 256
        assert info.grid * 2 * info.tile_m * 128 * 4 > SCRATCH_BYTES
        x = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
        y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        packed = torch.empty((hm.packed_size(hm.desc(2, n, k)),), dtype=torch.uint8, device="cuda")
        status = lib.hm_gemm_w4a16_noalloc(2, P(x.data_ptr()), P(packed.data_ptr()), P(y.data_ptr()), m, n, k,
                                           P(torch.cuda.current_stream().cuda_stream))
        assert status == 3                       # HM_ERR_WORKSPACE: nothing launched
    finally:
        for v, val in old.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val
    # formats other than W4A16 have no allocation-free entry
    assert lib.hm_gemm_w4a16_noalloc(3, P(x.data_ptr()), P(packed.data_ptr()), P(y.data_ptr()), 4, n, k,
                                     None) == 1
    torch.cuda.synchronize()
    assert hm.device_error() == 0
