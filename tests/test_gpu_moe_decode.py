"""GPU parity of the grouped decode kernel (warp-level MMA over every expert's 16-row token tiles,
the (tile, k-block) space cut into one range per SM) that serves W4A16 MoE layers with few rows per
expert, against the oracle's per-expert product over expert-sorted rows: every unit format, experts
larger than a token tile, empty experts, ragged N, ranges that split tiles across CTAs and cross
expert boundaries, the planner's default choice, determinism, and malformed offsets or headers."""
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


def experts(hm, fmt, e, n, k, has_zero=False, group=0, seed=0):
    """E experts quantized by the oracle and transformed one by one; returns (QuantWeights, packed
    tensors, device pointer array)."""
    qws, packs = [], []
    for i in range(e):
        zg = k if group == -1 else (group or 128)
        z = None
        if has_zero:   # u4 zero-points per group (INT8: u8 per 128-K block)
            z = np.random.default_rng(seed + 300 + i).integers(0, 256 if fmt == 7 else 16, size=(n, k // zg),
                                                                dtype=np.uint8)
        qw = QuantWeight(fmt, synth.weights(n, k, seed=seed + i), z, group=group)
        qws.append(qw)
        packs.append(qw.transform(hm)[1])
    ptrs = torch.tensor([p.data_ptr() for p in packs], dtype=torch.int64, device="cuda")
    return qws, packs, ptrs


def decode_case(hm, fmt, counts, n, k, has_zero=False, group=0, seed=0):
    e = len(counts)
    offsets = np.zeros(e + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    rows = int(offsets[-1])
    qws, _, ptrs = experts(hm, fmt, e, n, k, has_zero, group, seed)
    x = synth.activations(rows, k, seed=seed + 999)
    full, y = canary_out(rows, n)
    hm.moe_gemm(fmt, x.cuda(), torch.from_numpy(offsets).cuda(), ptrs, n, k, out=y)
    torch.cuda.synchronize()
    assert_close(y, og.moe_gemm(bf16_np(x), offsets, [q.what for q in qws]), f"moe decode fmt={fmt} counts={counts}")
    check_canary(full, rows, f"moe decode fmt={fmt}")
    assert hm.device_error() == 0
    return y


FORMATS = [(1, False, 0), (1, True, 0), (1, True, -1), (2, False, 0), (5, False, 0), (6, True, 32), (6, False, 64),
           (7, True, 0), (7, False, 0)]


@pytest.mark.parametrize("tokens", ["8", "16", "tc"])
@pytest.mark.parametrize("fmt,has_zero,group", FORMATS)
def test_every_unit_format(hm, fmt, has_zero, group, tokens, monkeypatch):
    """The warp-MMA decode kernel with token tiles of 8 and 16 rows, and the tensor-core decode
    kernel (INT4; the other formats keep the warp-MMA kernel); experts of 1 to 40 rows (up to five
    token tiles) and empty ones; 216 or more units over the SMs, so most tiles are split along K
    between CTAs."""
    monkeypatch.setenv("HM_MOE_GEMV", "1")
    monkeypatch.setenv("HM_DECODE_TC", "1" if tokens == "tc" else "0")
    if tokens != "tc":
        monkeypatch.setenv("HM_MOE_GEMV_TOKENS", tokens)
    decode_case(hm, fmt, [3, 0, 17, 40, 1, 0, 9, 16], 384, 1024, has_zero, group, seed=10 * fmt + 1)


@pytest.mark.parametrize("fmt", [1, 2])
def test_ragged_n_and_single_k_block(hm, fmt, monkeypatch):
    """N = 200 (the last weight tile is partly outside the matrix) and K = 128 (one unit per tile)."""
    monkeypatch.setenv("HM_MOE_GEMV", "1")
    decode_case(hm, fmt, [2, 5, 0, 1], 200, 128, fmt == 1, seed=5)


@pytest.mark.parametrize("tokens", ["8", "16", "tc"])
@pytest.mark.parametrize("fmt", [1, 7])
def test_ranges_cross_experts(hm, fmt, tokens, monkeypatch):
    """64 experts with Zipf top-4 routing of 24 tokens (96 rows): about 180 tiles of 16 k-blocks,
    so each CTA's range runs over several tiles and experts."""
    monkeypatch.setenv("HM_MOE_GEMV", "1")
    monkeypatch.setenv("HM_DECODE_TC", "1" if tokens == "tc" else "0")
    if tokens != "tc":
        monkeypatch.setenv("HM_MOE_GEMV_TOKENS", tokens)
    _, _, offsets = synth.moe_routing(tokens=24, experts=64, topk=4, seed=3)
    decode_case(hm, fmt, np.diff(offsets).tolist(), 512, 2048, fmt == 1, seed=7)


def test_default_choice_and_determinism(hm, capfd, monkeypatch):
    """At most two rows per expert on average: the planner takes the decode kernel by itself; two
    calls give identical bits; the tcgen05 kernel (HM_MOE_GEMV=0) agrees within the tolerance."""
    monkeypatch.setenv("HM_LOG", "1")
    _, _, offsets = synth.moe_routing(tokens=16, experts=64, topk=4, seed=4)
    n, k = 256, 1024
    qws, _, ptrs = experts(hm, 1, 64, n, k, True, seed=40)
    rows = int(offsets[-1])
    x = synth.activations(rows, k, seed=41).cuda()
    offs = torch.from_numpy(offsets).cuda()
    y1 = hm.moe_gemm(1, x, offs, ptrs, n, k)
    y2 = hm.moe_gemm(1, x, offs, ptrs, n, k)
    torch.cuda.synchronize()
    err = capfd.readouterr().err
    assert "kernel=decode" in err, err
    assert torch.equal(y1, y2)
    yref = og.moe_gemm(bf16_np(x), offsets, [q.what for q in qws])
    assert_close(y1, yref, "default decode")
    monkeypatch.setenv("HM_MOE_GEMV", "0")
    y3 = hm.moe_gemm(1, x, offs, ptrs, n, k)
    torch.cuda.synchronize()
    assert "kernel=tcgen05" in capfd.readouterr().err
    assert_close(y3, yref, "tcgen05 at the same size")
    assert hm.device_error() == 0


def test_no_workspace_runs_tcgen05(hm, capfd, monkeypatch):
    """Without a workspace the call takes the tcgen05 kernel, which needs none."""
    monkeypatch.setenv("HM_LOG", "1")
    n, k = 256, 512
    qws, _, ptrs = experts(hm, 2, 4, n, k, seed=50)
    offsets = np.array([0, 1, 1, 3, 4], dtype=np.int32)
    x = synth.activations(4, k, seed=51).cuda()
    y = torch.empty((4, n), dtype=torch.bfloat16, device="cuda")
    lib = hm.lib()
    import ctypes
    P = ctypes.c_void_p
    st = torch.cuda.current_stream().cuda_stream
    offs = torch.from_numpy(offsets).cuda()
    assert lib.hm_moe_gemm(2, P(x.data_ptr()), P(offs.data_ptr()), 4, P(ptrs.data_ptr()), P(y.data_ptr()), 4, n, k,
                           None, 0, P(st)) == 0
    torch.cuda.synchronize()
    assert "kernel=tcgen05" in capfd.readouterr().err
    assert_close(y, og.moe_gemm(bf16_np(x), offsets, [q.what for q in qws]), "no workspace")
    assert hm.device_error() == 0


def test_bad_offsets_store_nothing(hm, monkeypatch):
    monkeypatch.setenv("HM_MOE_GEMV", "1")
    n, k = 128, 256
    _, _, ptrs = experts(hm, 1, 2, n, k, seed=60)
    x = synth.activations(8, k, seed=61).cuda()
    y = torch.full((64, n), 7.0, dtype=torch.bfloat16, device="cuda")
    for offs in ([0, 6, 3], [0, 4, 100], [1, 4, 8]):
        hm.moe_gemm(1, x, torch.tensor(offs, dtype=torch.int32, device="cuda"), ptrs, n, k, out=y[:8])
        torch.cuda.synchronize()
        assert hm.device_error() & 4, offs
        assert (y == 7.0).all(), offs


def test_mismatched_header_stores_nothing(hm, monkeypatch):
    """An expert whose packed weight was made for another K: error bit 0, every CTA stops before
    reading any weight (the headers are checked in the set-up), nothing is stored."""
    monkeypatch.setenv("HM_MOE_GEMV", "1")
    n, k = 128, 256
    _, packs, _ = experts(hm, 1, 2, n, k, seed=70)
    other = QuantWeight(1, synth.weights(n, 2 * k, seed=71)).transform(hm)[1]
    ptrs = torch.tensor([packs[0].data_ptr(), other.data_ptr()], dtype=torch.int64, device="cuda")
    x = synth.activations(8, k, seed=72).cuda()
    y = torch.full((8, n), 7.0, dtype=torch.bfloat16, device="cuda")
    hm.moe_gemm(1, x, torch.tensor([0, 4, 8], dtype=torch.int32, device="cuda"), ptrs, n, k, out=y)
    torch.cuda.synchronize()
    assert hm.device_error() & 1
    assert (y == 7.0).all()


def test_rows_past_the_last_expert_untouched(hm, monkeypatch):
    """offsets[E] < rows: the trailing rows belong to no expert and keep their contents. (4 tiles of
    4 k-blocks: fewer units than SMs, so only the first 16 CTAs take one unit each and every tile is
    split four ways.)"""
    monkeypatch.setenv("HM_MOE_GEMV", "1")
    monkeypatch.setenv("HM_MOE_GEMV_TOKENS", "8")
    n, k = 256, 512
    qws, _, ptrs = experts(hm, 1, 3, n, k, seed=80)
    offsets = np.array([0, 2, 2, 5], dtype=np.int32)
    x = synth.activations(9, k, seed=81)
    y = torch.full((9, n), 7.0, dtype=torch.bfloat16, device="cuda")
    hm.moe_gemm(1, x.cuda(), torch.from_numpy(offsets).cuda(), ptrs, n, k, out=y)
    torch.cuda.synchronize()
    assert_close(y[:5], og.moe_gemm(bf16_np(x[:5]), offsets, [q.what for q in qws]), "leading rows")
    assert (y[5:] == 7.0).all()
    assert hm.device_error() == 0


def test_one_workspace_for_every_entry_and_size(hm, monkeypatch):
    """One zero-filled workspace, in stream order, for: a tcgen05 W4A16 GEMM whose tiles are split
    along K (partials of 64-token tiles), the W4A8 grouped GEMM that quantizes its activations into
    the workspace, the decode kernel with tiles split 24 ways (arrival counters in global memory),
    and the grouped decode kernel; then the first and third again. Every call's partials and
    activations lie after the counter block, so each matches the oracle."""
    from oracle import quant as oq
    from oracle.formats import decode_e4m3
    monkeypatch.setenv("HM_MOE_GEMV", "1")
    assert hm.plan(1, 256, 1024, 8192, torch.cuda.get_device_properties(0).multi_processor_count)["stream_k"] == 1
    lib = hm.lib()
    need = max(lib.hm_workspace_size(1, 256, 1024, 8192), lib.hm_workspace_size(1, 17, 640, 3072),
               lib.hm_moe_workspace_size(3, 64, 4, 512, 1024), lib.hm_moe_workspace_size(1, 86, 8, 384, 1024))
    ws = torch.zeros((need,), dtype=torch.uint8, device="cuda")

    def dense(m, n, k, seed):
        qw = QuantWeight(1, synth.weights(n, k, seed=seed), synth.zero_points(n, k // 128, seed=seed + 1))
        _, packed = qw.transform(hm)
        x = synth.activations(m, k, seed=seed + 2)
        return lambda: assert_close(hm.gemm(1, x.cuda(), packed, n, k, ws=ws), og.gemm(bf16_np(x), qw.what),
                                    f"dense {m}x{n}x{k}")

    big, small = dense(256, 1024, 8192, 90), dense(17, 640, 3072, 93)
    # W4A8 grouped, experts at a fixed stride, activations quantized inside the call
    counts = [20, 0, 30, 14]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    d0 = hm.desc(3, 512, 1024)
    buf = hm.alloc_moe_packed(d0, 4)
    qws = []
    for i in range(4):
        qw = QuantWeight(3, synth.weights(512, 1024, seed=100 + i))
        q, s, _ = qw.device_inputs()
        hm.transform(hm.desc(3, 512, 1024), q, s, None, out=hm.moe_expert_view(buf, d0, i))
        qws.append(qw)
    xa = synth.activations(64, 1024, seed=105, outlier_frac=0.01)
    xq, st = oq.quant_fp8_per_token(bf16_np(xa))
    ya_ref = og.moe_gemm(decode_e4m3(xq) * st[:, None], offsets, [q.what for q in qws])
    # grouped decode, W4A16 INT4 with a pointer list
    mcounts = [3, 0, 17, 40, 1, 0, 9, 16]
    moffs = np.concatenate([[0], np.cumsum(mcounts)]).astype(np.int32)
    mqws, _, ptrs = experts(hm, 1, 8, 384, 1024, True, seed=110)
    xm = synth.activations(86, 1024, seed=120)
    ym_ref = og.moe_gemm(bf16_np(xm), moffs, [q.what for q in mqws])

    big()
    ya = hm.moe_gemm_strided(3, xa.cuda(), torch.from_numpy(offsets).cuda(), buf, 4, hm.moe_stride(d0), 512, 1024,
                             ws=ws)
    assert_close(ya, ya_ref, "W4A8 grouped")
    small()
    ym = hm.moe_gemm(1, xm.cuda(), torch.from_numpy(moffs).cuda(), ptrs, 384, 1024, ws=ws)
    assert_close(ym, ym_ref, "grouped decode")
    big()
    small()
    assert hm.device_error() == 0
