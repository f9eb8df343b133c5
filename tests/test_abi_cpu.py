"""C-ABI checks that need no GPU: libhm.so loads, exports every function include/hm.h
declares, and its host-only queries and argument validation behave (no compute calls)."""
import ctypes
import os
import re

import pytest

from oracle import layout as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


def declared_functions():
    text = open(os.path.join(ROOT, "include", "hm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hm_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(hm):
    names = declared_functions()
    assert len(names) >= 15
    lib = ctypes.CDLL(hm.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


@pytest.mark.parametrize("fmt,n,k,hz", [(1, 4096, 4096, False), (1, 130, 256, True), (2, 256, 512, False),
                                        (3, 7168, 7168, False), (4, 8192, 8192, False), (4, 100, 64, False),
                                        (5, 4096, 14336, False), (5, 130, 128, False)])
def test_packed_size_matches_layout_spec(hm, fmt, n, k, hz):
    assert hm.packed_size(hm.desc(fmt, n, k, hz)) == L.packed_size(fmt, n, k, hz)


def test_packed_size_rejects_bad_shapes(hm):
    assert hm.packed_size(hm.desc(1, 128, 100)) == 0      # K not a multiple of 128
    assert hm.packed_size(hm.desc(4, 128, 96)) == 0       # NVFP4 K % 64
    assert hm.packed_size(hm.desc(2, 128, 128, True)) == 0  # zero-points only for INT4
    assert hm.packed_size(hm.desc(5, 128, 128, True)) == 0
    assert hm.packed_size(hm.desc(5, 128, 64)) == 0       # MXINT4 K % 128
    assert hm.packed_size(hm.desc(8, 128, 128)) == 0
    assert hm.packed_size(hm.desc(9, 128, 128)) == 0
    assert hm.packed_size(hm.desc(7, 130, 256)) == L.packed_size(7, 130, 256, False)
    assert hm.packed_size(hm.desc(7, 130, 256, True)) == L.packed_size(7, 130, 256, True)
    assert hm.packed_size(hm.desc(7, 130, 256, group=64)) == 0        # INT8 groups are 128
    # group sizes: INT4 takes multiples of 128 dividing K (or -1 per channel), format 6 takes 32 / 64
    assert hm.packed_size(hm.desc(1, 128, 512, group=256)) == L.packed_size(1, 128, 512, False)
    assert hm.packed_size(hm.desc(1, 128, 512, group=-1)) == L.packed_size(1, 128, 512, False)
    assert hm.packed_size(hm.desc(1, 128, 512, group=384)) == 0      # does not divide K
    assert hm.packed_size(hm.desc(1, 128, 512, group=64)) == 0       # below 128: format 6
    assert hm.packed_size(hm.desc(6, 128, 512, group=64)) == L.packed_size(6, 128, 512, False)
    assert hm.packed_size(hm.desc(6, 128, 512, True, group=32)) == L.packed_size(6, 128, 512, True)
    assert hm.packed_size(hm.desc(6, 128, 512, group=128)) == 0
    assert hm.packed_size(hm.desc(2, 128, 512, group=64)) == 0       # MX groups are 32
    # the GPTQ zero-point convention needs zero-points of an INT4 format
    assert hm.packed_size(hm.desc(1, 128, 512, True, zero_convention=1)) == L.packed_size(1, 128, 512, True)
    assert hm.packed_size(hm.desc(1, 128, 512, False, zero_convention=1)) == 0
    assert hm.packed_size(hm.desc(5, 128, 512, False, zero_convention=1)) == 0
    assert hm.packed_size(hm.desc(1, 128, 512, True, zero_convention=2)) == 0
    assert hm.packed_size(hm.desc(1, 0, 128)) == 0


def test_invalid_arguments_fail_before_any_launch(hm):
    lib = hm.lib()
    P = ctypes.c_void_p
    # null pointers / bad shapes are rejected on the host with HM_ERR_INVALID_ARG (1)
    assert lib.hm_gemm(1, None, None, None, None, None, 4, 256, 512, None, 0, None) == 1
    assert lib.hm_gemm(1, P(16), None, None, P(256), P(16), 4, 256, 100, P(256), 1 << 20, None) == 1
    assert lib.hm_gemm(9, P(16), None, None, P(256), P(16), 4, 256, 512, P(256), 1 << 20, None) == 1
    # misaligned packed pointer
    assert lib.hm_gemm(1, P(16), None, None, P(272), P(16), 4, 256, 512, P(256), 1 << 20, None) == 1
    # too small a workspace -> HM_ERR_WORKSPACE (3)
    assert lib.hm_gemm(1, P(16), None, None, P(256), P(16), 4, 256, 512, P(256), 16, None) == 3
    # M = 0 is a no-op
    assert lib.hm_gemm(1, None, None, None, None, None, 0, 256, 512, None, 0, None) == 0
    # MoE: unsupported format, bad expert count
    assert lib.hm_moe_gemm(3, P(16), P(16), 4, P(16), P(16), 8, 256, 512, None, 0, None) == 2
    assert lib.hm_moe_gemm(1, P(16), P(16), 0, P(16), P(16), 8, 256, 512, None, 0, None) == 1
    assert lib.hm_quant_act_fp8(P(16), 4, 100, P(16), P(16), None) == 1
    # SiLU-mul: inter a multiple of 8, rows >= 0, aligned non-null buffers; rows = 0 is a no-op
    assert lib.hm_silu_mul(P(16), P(16), 4, 12, None) == 1
    assert lib.hm_silu_mul(P(16), P(16), -1, 16, None) == 1
    assert lib.hm_silu_mul(None, P(16), 4, 16, None) == 1
    assert lib.hm_silu_mul(P(18), P(16), 4, 16, None) == 1
    assert lib.hm_silu_mul(None, None, 0, 16, None) == 0
    # 4 rows x (16 | 16) bf16 = 256 bytes in, 128 out: any overlap is refused before a CUDA call
    assert lib.hm_silu_mul(P(4096), P(4096), 4, 16, None) == 1
    assert lib.hm_silu_mul(P(4096), P(4096 + 240), 4, 16, None) == 1
    assert lib.hm_silu_mul(P(4096 + 112), P(4096), 4, 16, None) == 1
    assert lib.hm_quant_act_nvfp4(P(16), 4, 96, None, P(16), P(16), P(16), None, 0, None) == 1
    assert lib.hm_quant_act_nvfp4(P(16), 4, 128, None, P(16), P(16), P(16), None, 0, None) == 3


def test_plan_buckets(hm):
    seen = {}
    for m in (1, 16, 17, 64, 65, 256, 257, 1024, 1025, 8192):
        p = hm.plan(1, m, 4096, 4096, 152)
        seen[m] = p
        assert p["tile_n"] == 128 and p["tile_k"] == 128
        if m <= 32:   # decode-sized M: the warp-MMA decode kernel, built for 8, 16 or 32 tokens
            assert p["kernel"] == 1 and p["tile_m"] in (8, 16, 32) and p["tile_m"] >= m
        else:
            assert p["kernel"] == 0 and p["tile_m"] >= min(m, 16) and p["tile_m"] in (16, 32, 64, 128, 256)
        assert 1 <= p["grid"] <= 152
    assert [seen[m]["bucket"] for m in (1, 16, 17, 64, 65, 256, 257, 1024, 1025)] == [0, 0, 1, 1, 2, 2, 3, 3, 4]
    # M = 1: 32 tiles of 32 k-blocks, each cut into 4 K ranges (one per CTA)
    assert (seen[1]["stream_k"], seen[1]["grid"], seen[1]["tiles"]) == (1, 128, 32)
    assert seen[16]["stream_k"] == 1 and seen[16]["grid"] == 128   # M = 16 too: the decode kernel
    assert seen[8192]["stream_k"] == 0 and seen[8192]["tile_m"] == 256 and seen[8192]["tiles"] == 32 * 32
    assert seen[1024]["tile_m"] == 256 and seen[1024]["stream_k"] == 0   # 128 tiles cover 84 % of the SMs
    # 16 < M <= 512 (INT4): the cost model picks the measured-best (tile, stream-K) pair
    assert (seen[256]["tile_m"], seen[256]["stream_k"]) == (64, 0)     # 256 tiles cover the SMs
    assert (seen[64]["tile_m"], seen[64]["stream_k"]) == (32, 1)       # 64 tiles: split K
    p = hm.plan(1, 128, 4096, 4096, 152)
    assert (p["tile_m"], p["stream_k"], p["grid"]) == (64, 1, 128)   # 64 tiles, each cut in 2 K ranges
    p = hm.plan(1, 256, 4096, 14336, 152)
    assert (p["tile_m"], p["stream_k"]) == (128, 1)                  # long K: 128-token tiles, split
    # long K: stream-K; wide N: the 256-token tile from M = 256 on
    p = hm.plan(1, 128, 4096, 14336, 152)
    assert (p["tile_m"], p["stream_k"]) == (64, 1)
    assert hm.plan(1, 256, 14336, 4096, 152)["tile_m"] == 256
    assert hm.plan(1, 64, 14336, 4096, 152)["stream_k"] == 0           # 112 tiles of 64 tokens
    # every stream-K CTA gets at least one k-block
    p = hm.plan(1, 1, 128, 256, 152)
    assert p["grid"] == 2


def test_workspace_sizes(hm):
    for fmt in (1, 2, 3, 4):
        assert hm.workspace_size(fmt, 16, 4096, 4096) > 0
    # the internal activation buffers are included for the A8/A4 formats
    assert hm.workspace_size(3, 1024, 4096, 4096) >= 1024 * 4096 + hm.workspace_size(1, 1024, 4096, 4096) // 2
    assert hm.lib().hm_act_scale_size(130, 128) == L.act_scale_bytes(130, 128)


def test_status_strings(hm):
    lib = hm.lib()
    assert lib.hm_status_string(0) == b"ok"
    assert b"workspace" in lib.hm_status_string(3)
    assert hm.version().startswith("hm ")


def test_plan_block_scaled_two_ctas_per_sm(hm):
    """W4A8/W4A4 run two CTAs per SM: tile-parallel from four waves of tiles up, stream-K below
    (balanced CTAs), and one CTA per SM when tiles are fewer than SMs with tiles wider than 16."""
    for fmt in (3, 4):
        big = hm.plan(fmt, 8192, 8192, 8192, 152)          # 64 x 64 tiles
        assert big["stream_k"] == 0 and big["grid"] == 2 * 152 and big["tile_m"] == 128
        mid = hm.plan(fmt, 1024, 8192, 8192, 152)          # 8 x 64 = 512 tiles: tile-parallel
        assert mid["stream_k"] == 0 and mid["grid"] == 2 * 152
        tiny = hm.plan(fmt, 16, 8192, 8192, 152)           # 64 tiles of 16 tokens: stream-K,
        assert tiny["stream_k"] == 1 and tiny["grid"] == 64 * 4 and tiny["tile_m"] == 16   # 4 K ranges each
    # W4A8 at M = 128: the widest tile giving >= 1.4x SMs tiles (32 tokens: 4 x 64 = 256 tiles)
    p = hm.plan(3, 128, 8192, 8192, 152)
    assert p["tile_m"] == 32 and p["stream_k"] == 0 and p["grid"] == 256
    # W4A4 keeps 128-token tiles (its activation scale atoms hold 128 rows), tile-parallel
    p = hm.plan(4, 128, 8192, 8192, 152)
    assert p["tile_m"] == 128 and p["stream_k"] == 0 and p["grid"] == 64
    # too few tiles even at 32 tokens: stream-K, one CTA per SM (112 tiles: one K range each)
    p = hm.plan(3, 64, 7168, 7168, 152)
    assert p["tile_m"] == 32 and p["stream_k"] == 1 and p["grid"] == 112
    # W4A16 keeps one CTA per SM
    assert hm.plan(1, 8192, 8192, 8192, 152)["grid"] == 152
    # stream-K partials are sized for the widest grid the planner can choose
    assert hm.workspace_size(3, 16, 8192, 8192) >= 2 * 256 * 2 * 16 * 128 * 4


def test_plan_small_token_stages(hm):
    """INT4 token tiles 16/32 report the small-token kernel's load stages; HM_F16_SMALL=0 the general kernel's."""
    a = hm.plan(1, 24, 4096, 4096, 152)["stages"]
    os.environ["HM_F16_SMALL"] = "0"
    try:
        b = hm.plan(1, 24, 4096, 4096, 152)["stages"]
    finally:
        del os.environ["HM_F16_SMALL"]
    assert a >= 3 and b >= 2


def test_oversized_schedule_rejected(hm):
    """Problems whose (tile, k-block) space reaches 2^31 iterations are refused before any launch
    (the kernels index it in 32 bits)."""
    with pytest.raises(hm.HmError) as e:
        hm.plan(1, 1 << 22, 1 << 20, 1 << 16, 152)
    assert e.value.status == 2


def test_plan_decode_kernel(hm, monkeypatch):
    """W4A16 formats at M <= 32 take the warp-MMA decode kernel (built for 8, 16 or 32 tokens);
    with HM_DECODE_TC=1, INT4 up to 16 tokens takes the tensor-core decode kernel (16-token tiles);
    the block-scaled formats and M > 32 keep tcgen05; HM_GEMV=0 keeps tcgen05 for every M."""
    for fmt in (1, 2, 5):
        tiles = [hm.plan(fmt, m, 4096, 4096, 152)["tile_m"] for m in range(1, 33)]
        assert tiles == [8] * 8 + [16] * 8 + [32] * 16
        assert all(hm.plan(fmt, m, 4096, 4096, 152)["kernel"] == 1 for m in range(1, 33))
        assert hm.plan(fmt, 33, 4096, 4096, 152)["kernel"] == 0
    monkeypatch.setenv("HM_DECODE_TC", "1")
    assert [hm.plan(1, m, 4096, 4096, 152)["tile_m"] for m in range(1, 33)] == [16] * 16 + [32] * 16
    assert [hm.plan(1, m, 4096, 4096, 152)["kernel"] for m in range(1, 33)] == [2] * 16 + [1] * 16
    assert hm.plan(2, 1, 4096, 4096, 152)["kernel"] == 1   # INT4 only
    monkeypatch.delenv("HM_DECODE_TC")
    # 17..32 tokens on the 14336-wide layer: 112 whole tiles for tcgen05, which INT4 keeps;
    # MXFP4 always takes the decode kernel up to 32 tokens
    assert hm.plan(1, 32, 14336, 4096, 152)["kernel"] == 0
    assert hm.plan(1, 16, 14336, 4096, 152)["kernel"] == 1
    assert hm.plan(2, 32, 14336, 4096, 152)["kernel"] == 1
    assert hm.plan(5, 32, 14336, 4096, 152)["kernel"] == 1   # MXINT4 as MXFP4
    monkeypatch.setenv("HM_GEMV", "2")
    assert hm.plan(1, 32, 14336, 4096, 152)["kernel"] == 1
    # HM_SK_ALIGN=0: ranges across tile boundaries, one per SM (never more CTAs than units)
    monkeypatch.setenv("HM_SK_ALIGN", "0")
    p = hm.plan(1, 1, 14336, 4096, 152)
    assert (p["grid"], p["stream_k"]) == (152, 1)
    assert hm.plan(1, 1, 128, 256, 152)["grid"] == 2
    monkeypatch.delenv("HM_SK_ALIGN")
    for fmt in (3, 4):
        assert hm.plan(fmt, 1, 4096, 4096, 152)["kernel"] == 0
    # 152 tiles of two 128-K blocks on 152 SMs: one whole tile per CTA, no split
    p = hm.plan(1, 1, 152 * 128, 256, 152)
    assert (p["grid"], p["stream_k"]) == (152, 0)
    # two units: two CTAs
    p = hm.plan(1, 3, 200, 128, 152)
    assert (p["grid"], p["tiles"], p["stream_k"]) == (2, 2, 0)
    # tiles <= SMs: every tile cut into the same number of K ranges, one per CTA
    for n, k, grid, sk in ((14336, 4096, 112, 0), (4096, 14336, 128, 1), (1024, 1024, 64, 1), (640, 3072, 120, 1)):
        p = hm.plan(1, 1, n, k, 152)
        assert (p["grid"], p["stream_k"]) == (grid, sk), (n, k, p)
    # more tiles than SMs: one range per SM
    assert hm.plan(1, 1, 304 * 128, 256, 152)["grid"] == 152
    monkeypatch.setenv("HM_GEMV", "0")
    assert hm.plan(1, 1, 4096, 4096, 152)["kernel"] == 0
    assert hm.plan(1, 1, 4096, 4096, 152)["tile_m"] == 16


def test_workspace_holds_decode_counters(hm):
    """The decode kernel keeps 8 arrival counters per 128-row tile and tokens x 128 fp32 partials
    per CTA; the workspace for M <= 32 has room for both on any device up to the sizing limit."""
    n, k = 19456, 4096
    for m in (16, 32):
        assert hm.workspace_size(1, m, n, k) >= (n // 128) * 8 * 4 + 148 * m * 128 * 4


def test_plan_stream_k_equal_ranges(hm, monkeypatch):
    """tcgen05 stream-K with no more tiles than CTAs cuts every tile into the same number of K
    ranges (one per CTA); HM_SK_ALIGN=0 keeps ranges that run across tile boundaries."""
    p = hm.plan(3, 1, 7168, 7168, 152)              # 56 tiles, 304 CTA slots: 5 ranges per tile
    assert (p["stream_k"], p["grid"]) == (1, 280)
    p = hm.plan(1, 64, 4096, 4096, 152)             # 64 tiles of 32 tokens: 2 ranges per tile
    assert (p["tile_m"], p["stream_k"], p["grid"]) == (32, 1, 128)
    monkeypatch.setenv("HM_SK_ALIGN", "0")
    assert hm.plan(3, 1, 7168, 7168, 152)["grid"] == 304
    assert hm.plan(1, 64, 4096, 4096, 152)["grid"] == 152


def test_workspace_covers_every_plan(hm):
    """For any device up to the sizing limit, the workspace hm_workspace_size asks for holds the
    split partials and arrival counters of the plan hm_plan chooses (decode kernel: grid x tokens x
    128 fp32 partials and 8 counters per tile; tcgen05, including the block-scaled kernels' two CTAs
    per SM: grid x 2 x tile_m x 128 and 4 per tile)."""
    import random
    rng = random.Random(7)
    shapes = [(1, m, n, k) for m in (1, 8, 16, 17, 32, 33, 64, 200) for n, k in ((4096, 4096), (20480, 1024), (200, 128))]
    for _ in range(80):
        fmt = rng.choice((1, 2, 3, 4, 5))
        shapes.append((fmt, rng.randint(1, 300), 128 * rng.randint(1, 200) - rng.choice((0, 2, 64)), 256 * rng.randint(1, 30)))
    for fmt, m, n, k in shapes:
        ws = hm.workspace_size(fmt, m, n, k)
        for sms in (1, 2, 7, 64, 148, 152, 160, 256):
            p = hm.plan(fmt, m, n, k, sms)
            if p["kernel"] in (1, 2):
                need = p["grid"] * p["tile_m"] * 128 * 4 + p["tiles"] * 8 * 4
            else:
                need = (p["grid"] * 2 * p["tile_m"] * 128 * 4 if p["stream_k"] else 0) + p["tiles"] * 4 * 4
            assert ws >= need, (fmt, m, n, k, sms, p, ws, need)


def test_plan_log_line(hm):
    """HM_LOG=1 prints the configuration each planned call takes (stderr), nothing otherwise."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = "from moe_hm_gemm_gb300 import hm; hm.plan(1, 1, 14336, 4096, 152); hm.plan(4, 8192, 8192, 8192, 152)"
    env = dict(os.environ, HM_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, check=True)
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("[hm] ")]
    assert len(lines) == 2
    assert "fmt=1 M=1 N=14336 K=4096 kernel=decode tile_m=8" in lines[0]
    assert "fmt=4 M=8192 N=8192 K=8192 kernel=tcgen05 tile_m=128 tile_k=256" in lines[1]
    env.pop("HM_LOG")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, check=True)
    assert "[hm]" not in r.stderr


def test_binding_rejects_host_and_strided_tensors(hm):
    """The binding hands raw pointers to the C ABI, so it refuses host tensors, strided views and
    mis-shaped outputs before any call."""
    import torch
    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    packed = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError):
        hm.gemm(1, x, packed, 128, 256)
    with pytest.raises(ValueError):
        hm.gemm_noalloc(1, x, packed, 128, 256)
    with pytest.raises(ValueError):
        hm.moe_gemm(1, x, torch.zeros(3, dtype=torch.int32), torch.zeros(2, dtype=torch.int64), 128, 256)
    with pytest.raises(ValueError):
        hm.quant_act_fp8(x)
    with pytest.raises(ValueError):
        hm.quant_act_nvfp4(x[:, ::2])
    with pytest.raises(ValueError):
        hm.quantize_weight(hm.desc(1, 128, 256), torch.zeros((128, 256)))
    with pytest.raises(ValueError):
        hm.transform(hm.desc(1, 128, 256), packed, packed)
    with pytest.raises(ValueError):
        hm.dequant(hm.desc(1, 128, 256), packed)


def test_plan_invariants_random(hm):
    """For random formats, shapes and SM counts the plan satisfies what the kernels rely on: every
    CTA holds at least one k-block (grid <= tiles x k-blocks), at most one CTA per SM for W4A16 and
    two for the block-scaled kernels, tiles = token tiles x 128-row tiles, the decode kernel only for
    W4A16 formats at M <= 32 with a token tile covering M, token tiles the kernels are built for, a
    split flag whenever CTAs share a tile, and at least two pipeline stages."""
    import random
    rng = random.Random(11)
    for _ in range(3000):
        fmt = rng.choice((1, 2, 3, 4, 5))
        m = rng.choice((1, 2, 8, 15, 16, 17, 31, 32, 33, 64, 100, 256, 1000, 4096, 9000))
        n = 128 * rng.randint(1, 160) - rng.choice((0, 2, 64))
        k = (256 if fmt == 4 else 128) * rng.randint(1, 60)
        sms = rng.choice((1, 2, 7, 64, 148, 152, 160, 256))
        p = hm.plan(fmt, m, n, k, sms)
        n_tiles = -(-n // 128)
        kb_total = k // p["tile_k"]
        assert p["tile_k"] == (256 if fmt == 4 else 128)
        assert p["stages"] >= 2
        if p["kernel"] == 1:
            assert fmt in (1, 2, 5) and m <= 32 and p["tile_m"] in (8, 16, 32) and p["tile_m"] >= m
            assert p["tiles"] == n_tiles
        elif p["kernel"] == 2:
            assert fmt == 1 and m <= 16 and p["tile_m"] == 16 and p["tiles"] == n_tiles
        else:
            assert p["tile_m"] in ((16, 32, 64, 128) if fmt in (3, 4) else (16, 32, 64, 128, 256))
            assert p["tiles"] == -(-m // p["tile_m"]) * n_tiles
            if fmt == 4 and m > 16:
                assert p["tile_m"] == 128          # its activation scale atoms hold 128 rows
        per_sm = 2 if fmt in (3, 4) and p["kernel"] == 0 else 1
        assert 1 <= p["grid"] <= sms * per_sm
        assert p["grid"] <= p["tiles"] * kb_total, (fmt, m, n, k, sms, p)
        if p["grid"] > p["tiles"]:
            assert p["stream_k"] == 1
        # stream-K covers sk_tiles leading tiles with non-empty ranges; the rest run in full waves
        assert (p["sk_tiles"] > 0) == (p["stream_k"] == 1)
        if p["stream_k"]:
            assert 1 <= p["sk_tiles"] <= p["tiles"] and p["grid"] <= p["sk_tiles"] * kb_total, (fmt, m, n, k, sms, p)
            if p["sk_tiles"] < p["tiles"]:
                assert fmt in (1, 2, 5) and p["kernel"] == 0 and p["tile_m"] >= 128
                assert (p["tiles"] - p["sk_tiles"]) % p["grid"] == 0 and p["sk_tiles"] < p["grid"]


def test_plan_hybrid_waves(hm, monkeypatch):
    """W4A16 with more whole tiles than CTAs: the tiles a last partial wave would hold (tiles mod
    grid) run as stream-K ranges first, by default for K loops of 64+ blocks with a remainder of at
    most half a wave; HM_SK_HYBRID=1 up to 90 % of a wave, HM_SK_HYBRID=0 never; either
    HM_STREAM_K value leaves it out (whole waves, or plain stream-K)."""
    p = hm.plan(1, 4096, 4096, 14336, 152)    # 512 tiles of 112 k-blocks: 3 waves + 56
    assert (p["tile_m"], p["stream_k"], p["sk_tiles"], p["grid"], p["tiles"]) == (256, 1, 56, 152, 512)
    p = hm.plan(5, 4096, 4096, 14336, 152)    # MXINT4 restored weights: the same kernel and schedule
    assert (p["stream_k"], p["sk_tiles"]) == (1, 56)
    assert hm.plan(1, 8192, 4096, 14336, 152)["stream_k"] == 0      # remainder 112 of 152: whole waves
    assert hm.plan(1, 4096, 4096, 4096, 152)["stream_k"] == 0       # 32 k-blocks per tile: whole waves
    assert hm.plan(3, 4096, 7168, 7168, 152)["sk_tiles"] == 0      # block-scaled: its own schedule
    monkeypatch.setenv("HM_SK_HYBRID", "1")
    p = hm.plan(1, 4096, 4096, 4096, 152)     # 512 tiles: 3 waves + 56
    assert (p["tile_m"], p["stream_k"], p["sk_tiles"], p["grid"], p["tiles"]) == (256, 1, 56, 152, 512)
    p = hm.plan(1, 8192, 14336, 4096, 152)    # 3584 tiles: 23 waves + 88
    assert (p["stream_k"], p["sk_tiles"]) == (1, 88)
    p = hm.plan(1, 1024, 14336, 4096, 152)    # 448 tiles: 2 waves + 144 (95 % of a wave): whole waves
    assert (p["stream_k"], p["sk_tiles"], p["grid"]) == (0, 0, 152)
    p = hm.plan(1, 1024, 4096, 4096, 152)     # 128 tiles: one partial wave, tile-parallel
    assert (p["stream_k"], p["sk_tiles"], p["grid"]) == (0, 0, 128)
    monkeypatch.setenv("HM_SK_HYBRID", "0")
    assert hm.plan(1, 4096, 4096, 14336, 152)["stream_k"] == 0
    monkeypatch.delenv("HM_SK_HYBRID")
    monkeypatch.setenv("HM_STREAM_K", "0")
    assert hm.plan(1, 4096, 4096, 14336, 152)["stream_k"] == 0
    monkeypatch.setenv("HM_STREAM_K", "1")
    p = hm.plan(1, 4096, 4096, 14336, 152)
    assert (p["stream_k"], p["sk_tiles"]) == (1, 512)


def test_moe_gather_combine_argument_checks(hm):
    lib = hm.lib()
    P = ctypes.c_void_p
    # gather: K % 8, negative sizes, null or misaligned pointers -> HM_ERR_INVALID_ARG; rows = 0 no-op
    assert lib.hm_moe_gather(P(16), P(16), P(4096), 4, 8, 12, None) == 1
    assert lib.hm_moe_gather(P(16), P(16), P(4096), -1, 8, 16, None) == 1
    assert lib.hm_moe_gather(None, P(16), P(4096), 4, 8, 16, None) == 1
    assert lib.hm_moe_gather(P(24), P(16), P(4096), 4, 8, 16, None) == 1
    assert lib.hm_moe_gather(P(16), P(18), P(4096), 4, 8, 16, None) == 1
    assert lib.hm_moe_gather(None, None, None, 4, 0, 16, None) == 0
    # combine: N % 8, topk < 1, misaligned y / out / pos / w -> HM_ERR_INVALID_ARG; T = 0 no-op
    assert lib.hm_moe_combine(P(16), P(16), P(16), P(4096), 4, 8, 32, 12, None) == 1
    assert lib.hm_moe_combine(P(16), P(16), P(16), P(4096), 4, 0, 32, 16, None) == 1
    assert lib.hm_moe_combine(P(24), P(16), P(16), P(4096), 4, 8, 32, 16, None) == 1
    assert lib.hm_moe_combine(P(16), P(16), P(18), P(4096), 4, 8, 32, 16, None) == 1
    assert lib.hm_moe_combine(P(16), None, P(16), P(4096), 4, 8, 32, 16, None) == 1
    assert lib.hm_moe_combine(None, None, None, None, 0, 8, 32, 16, None) == 0


def test_mma_peak_probe_argument_checks(hm):
    lib = hm.lib()
    fl = ctypes.c_double(0.0)
    assert lib.hm_mma_peak_probe(7, 10, ctypes.byref(fl), None) == 1
    assert lib.hm_mma_peak_probe(0, 0, ctypes.byref(fl), None) == 1
    assert lib.hm_mma_peak_probe(0, 10, None, None) == 1


def test_moe_strided_argument_checks(hm):
    lib = hm.lib()
    P = ctypes.c_void_p
    st = hm.moe_stride(hm.desc(3, 256, 512))
    # stride not a multiple of 256, or smaller than one packed weight
    assert lib.hm_moe_gemm_strided(3, P(256), None, P(256), 2, P(256), st + 16, P(256), 8, 256, 512, None, 0, None) == 1
    assert lib.hm_moe_gemm_strided(3, P(256), None, P(256), 2, P(256), 256, P(256), 8, 256, 512, None, 0, None) == 1
    # misaligned packed buffer, zero experts
    assert lib.hm_moe_gemm_strided(3, P(256), None, P(256), 2, P(272), st, P(256), 8, 256, 512, None, 0, None) == 1
    assert lib.hm_moe_gemm_strided(3, P(256), None, P(256), 0, P(256), st, P(256), 8, 256, 512, None, 0, None) == 1
    # W4A4 takes bf16 activations only; too many experts for the block-scaled kernel
    st4 = hm.moe_stride(hm.desc(4, 256, 512))
    assert lib.hm_moe_gemm_strided(4, P(256), P(256), P(256), 2, P(256), st4, P(256), 8, 256, 512, None, 0, None) == 2
    assert lib.hm_moe_gemm_strided(3, P(256), None, P(256), 300, P(256), st, P(256), 8, 256, 512, None, 0, None) == 2
    # internal activation quantization needs the workspace
    assert lib.hm_moe_workspace_size(3, 8, 2, 256, 512) >= 8 * 512 + 8 * 4
    assert lib.hm_moe_gemm_strided(3, P(256), None, P(256), 2, P(256), st, P(256), 8, 256, 512, None, 0, None) == 3
    # W4A16: the grouped decode kernel's fp32 partials (up to 256 CTAs x 16 tokens x 128 rows) and
    # 8 counters per (token tile, weight tile), at most rows / 16 + 1 + min(E, rows) token tiles;
    # more than 256 experts run the tcgen05 kernel only, which needs none
    assert lib.hm_moe_workspace_size(1, 8, 2, 256, 512) >= 256 * 16 * 128 * 4 + (0 + 1 + 2) * 2 * 8 * 4
    assert lib.hm_moe_workspace_size(7, 8, 2, 256, 512) == lib.hm_moe_workspace_size(1, 8, 2, 256, 512)
    assert lib.hm_moe_workspace_size(1, 8, 300, 256, 512) == 0
    # rows = 0 is a no-op
    assert lib.hm_moe_gemm_strided(3, None, None, None, 2, None, st, None, 0, 256, 512, None, 0, None) == 0
