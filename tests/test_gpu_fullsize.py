"""GPU parity at the benchmarked full sizes, on sampled outputs the oracle computes one by one:
the grouped MoE gate-up (N = 4096, K = 7168) and down (N = 7168, K = 2048) layers (E = 256,
T = 16384 and 16 tokens with top-8 Zipf(1.1) routing) in the W4A16 formats, and the dense MXINT4 layer
14336 x 4096 at M = 1 and 8192.

The weights and activations come from the seeded device generators the benchmark uses; the
oracle quantizes host copies of the sampled weight rows itself (quantization is row-local), so no
oracle input comes from the library's kernels."""
import numpy as np
import pytest
import torch

from moe_hm_gemm_gb300 import synth
from oracle import gemm as og
from oracle import quant as oq

from .gpu_util import bf16_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


def restore_rows(fmt, w_rows, z_rows):
    """Oracle restore of whole weight rows (float64 [S, K]) quantized by the oracle."""
    if fmt == 1:
        q, s = oq.quant_int4(w_rows, zeros=z_rows)
        return oq.dequant_int4(q, s, z_rows)
    if fmt == 2:
        return oq.dequant_mxfp4(*oq.quant_mxfp4(w_rows))
    return oq.dequant_mxint4(*oq.quant_mxint4(w_rows))


@pytest.mark.parametrize("t", [16384, 16])
@pytest.mark.parametrize("layer", ["gate_up", "down"])
@pytest.mark.parametrize("fmt", [1, 2, 5])
def test_moe_full_size_sampled(hm, fmt, layer, t):
    """T = 16384 runs the grouped tcgen05 kernel, T = 16 (128 rows over 256 experts) the grouped
    decode kernel."""
    e = 256
    n, k = (4096, 7168) if layer == "gate_up" else (7168, 2048)
    _, expert_of_row, offsets = synth.moe_routing(t, experts=e, topk=8, seed=0)
    rows = int(offsets[-1])
    rng = np.random.default_rng(5)
    rs = rng.integers(0, rows, size=256)
    ns = rng.integers(0, n, size=256)
    need = {}
    for i, r in enumerate(rs):
        need.setdefault(int(expert_of_row[r]), []).append(i)
    d = hm.desc(fmt, n, k, fmt == 1)
    packs, w_rows, z_rows = [], np.zeros((256, k)), np.zeros((256, k // 128), dtype=np.int64)
    for ei in range(e):
        w = synth.device_weights(n, k, seed=10000 + ei)
        z = synth.device_zero_points(n, k // 128, seed=20000 + ei) if fmt == 1 else None
        q, s, _ = hm.quantize_weight(d, w, z)
        packs.append(hm.transform(d, q, s, z))
        for i in need.get(ei, []):
            w_rows[i] = w[int(ns[i])].cpu().numpy()
            if z is not None:
                z_rows[i] = z[int(ns[i])].cpu().numpy()
        del w, q, s
    ptrs = torch.tensor([p.data_ptr() for p in packs], dtype=torch.int64, device="cuda")
    x = synth.device_activations(rows, k, seed=30000 + t)
    y = hm.moe_gemm(fmt, x, torch.from_numpy(offsets).cuda(), ptrs, n, k)
    torch.cuda.synchronize()
    what = restore_rows(fmt, w_rows, z_rows if fmt == 1 else None)
    xs = bf16_np(x[torch.from_numpy(rs).cuda()])
    ref = np.einsum("ik,ik->i", xs, what)
    got = bf16_np(y[torch.from_numpy(rs).cuda(), torch.from_numpy(ns).cuda()])
    ok = og.tolerance_ok(got, ref)
    assert ok.all(), f"fmt={fmt}: {int((~ok).sum())} of 256 sampled outputs outside tolerance"
    assert hm.device_error() == 0


def test_mxint4_dense_full_size_sampled(hm):
    n, k = 14336, 4096
    w = synth.weights(n, k, seed=1)
    q, e = oq.quant_mxint4(w)
    from .gpu_util import pack_nibbles
    d = hm.desc(5, n, k)
    packed = hm.transform(d, torch.from_numpy(pack_nibbles(q)).cuda(), torch.from_numpy(e.astype(np.uint8)).cuda())
    rng = np.random.default_rng(0)
    for m in (1, 8192):
        x = synth.activations(m, k, seed=3)
        y = hm.gemm(5, x.cuda(), packed, n, k)
        torch.cuda.synchronize()
        ms = rng.integers(0, m, size=256)
        ns = rng.integers(0, n, size=256)
        ref = np.einsum("ik,ik->i", bf16_np(x[torch.from_numpy(ms)]), oq.dequant_mxint4(q[ns], e[ns]))
        got = bf16_np(y.cpu()[torch.from_numpy(ms), torch.from_numpy(ns)])
        ok = og.tolerance_ok(got, ref)
        assert ok.all(), f"M={m}: {int((~ok).sum())} sampled outputs outside tolerance"
    assert hm.device_error() == 0
