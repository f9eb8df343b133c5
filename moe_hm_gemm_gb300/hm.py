"""Python binding of libhm.so (include/hm.h): argument marshalling only.

Every function takes torch tensors (device memory owned by the caller), passes their
pointers and sizes to the C ABI on the current CUDA stream, and raises HmError on a
non-OK status. No computation happens here; if the shared library is missing the import
fails loudly (there is no fallback).
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhm.so")

W4A16_INT4, W4A16_MXFP4, W4A8_MXFP4, W4A4_NVFP4, W4A16_MXINT4, W4A16_INT4_G32, W8A16_INT8 = 1, 2, 3, 4, 5, 6, 7
FORMATS = {"w4a16_int4": W4A16_INT4, "w4a16_mxfp4": W4A16_MXFP4,
           "w4a8_mxfp4": W4A8_MXFP4, "w4a4_nvfp4": W4A4_NVFP4, "w4a16_mxint4": W4A16_MXINT4,
           "w4a16_int4_g32": W4A16_INT4_G32, "w8a16_int8": W8A16_INT8}
ZP_INT, ZP_GPTQ = 0, 1


class HmError(RuntimeError):
    def __init__(self, status, where):
        super().__init__(f"{where}: {_lib.hm_status_string(status).decode()} (status {status})")
        self.status = status


class WeightDesc(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("has_zero", ctypes.c_int32), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("tensor_scale", ctypes.c_float), ("group", ctypes.c_int32),
                ("zero_convention", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("bucket", "tile_m", "tile_n", "tile_k", "stages", "stream_k", "grid", "tiles", "kernel",
                 "sk_tiles")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libhm.so not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, SZ, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    D = ctypes.POINTER(WeightDesc)
    sig = {
        "hm_packed_size": (SZ, [D]),
        "hm_quantize_workspace_size": (SZ, [D]),
        "hm_quantize_weight": (I32, [D, P, P, P, P, P, P, SZ, P]),
        "hm_transform": (I32, [D, P, P, P, P, P]),
        "hm_dequant": (I32, [D, P, P, P]),
        "hm_quant_act_fp8": (I32, [P, I64, I64, P, P, P]),
        "hm_silu_mul": (I32, [P, P, I64, I64, P]),
        "hm_moe_gather": (I32, [P, P, P, I64, I64, I64, P]),
        "hm_moe_combine": (I32, [P, P, P, P, I64, I32, I64, I64, P]),
        "hm_act_scale_size": (SZ, [I64, I64]),
        "hm_act_workspace_size": (SZ, [I64, I64]),
        "hm_quant_act_nvfp4": (I32, [P, I64, I64, P, P, P, P, P, SZ, P]),
        "hm_workspace_size": (SZ, [I32, I64, I64, I64]),
        "hm_gemm": (I32, [I32, P, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "hm_moe_gemm": (I32, [I32, P, P, I32, P, P, I64, I64, I64, P, SZ, P]),
        "hm_moe_workspace_size": (SZ, [I32, I64, I32, I64, I64]),
        "hm_moe_gemm_strided": (I32, [I32, P, P, P, I32, P, I64, P, I64, I64, I64, P, SZ, P]),
        "hm_gemm_w4a16_noalloc": (I32, [I32, P, P, P, I64, I64, I64, P]),
        "hm_plan": (I32, [I32, I64, I64, I64, I32, ctypes.POINTER(PlanInfo)]),
        "hm_get_device_error": (ctypes.c_uint32, [P]),
        "hm_debug_wait_timeout": (I32, [ctypes.c_uint64, P]),
        "hm_mma_peak_probe": (I32, [I32, I32, ctypes.POINTER(ctypes.c_double), P]),
        "hm_set_trace_buffer": (I32, [P, SZ]),
        "hm_status_string": (ctypes.c_char_p, [I32]),
        "hm_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _ = F
    return lib


_lib = _load()


def lib():
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(*named):
    """The C ABI takes raw device pointers: every tensor passed must be a contiguous CUDA tensor
    (None is passed through as NULL). Raises ValueError otherwise."""
    for name, t in named:
        if t is not None and (not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name}: expected a contiguous CUDA tensor")


def _out(y, shape, name="out"):
    """An output tensor given by the caller: contiguous CUDA bf16 of exactly `shape`."""
    _dev((name, y))
    if y.dtype != torch.bfloat16 or tuple(y.shape) != tuple(shape):
        raise ValueError(f"{name}: expected bf16 {tuple(shape)}, got {y.dtype} {tuple(y.shape)}")
    return y


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status, where):
    if status != 0:
        raise HmError(status, where)


def desc(fmt, n, k, has_zero=False, tensor_scale=1.0, group=0, zero_convention=ZP_INT):
    return WeightDesc(int(fmt), int(bool(has_zero)), int(n), int(k), float(tensor_scale), int(group),
                      int(zero_convention))


def group_of(d):
    """K values per scale of a description (its `group`, or the format's own for 0; -1 = K)."""
    if d.group == -1:
        return d.K
    if d.group:
        return d.group
    return {W4A16_INT4: 128, W4A16_INT4_G32: 32, W4A4_NVFP4: 16, W8A16_INT8: 128}.get(d.fmt, 32)


def packed_size(d):
    return _lib.hm_packed_size(ctypes.byref(d))


def quantize_weight(d, w, zeros=None):
    """fp32 W [N,K] (device) -> (q [N,K/2] uint8, scales, g) in the standard format."""
    _dev(("w", w), ("zeros", zeros))
    if w.dtype != torch.float32:
        raise ValueError("w: expected float32")
    dev = w.device
    q = torch.empty((d.N, d.K if d.fmt == W8A16_INT8 else d.K // 2), dtype=torch.uint8, device=dev)
    if d.fmt in (W4A16_INT4, W4A16_INT4_G32, W8A16_INT8):
        scales = torch.empty((d.N, d.K // group_of(d)), dtype=torch.bfloat16, device=dev)
    elif d.fmt in (W4A16_MXFP4, W4A8_MXFP4, W4A16_MXINT4):
        scales = torch.empty((d.N, d.K // 32), dtype=torch.uint8, device=dev)
    else:
        scales = torch.empty((d.N, d.K // 16), dtype=torch.uint8, device=dev)
    g = torch.empty((1,), dtype=torch.float32, device=dev)
    wsz = _lib.hm_quantize_workspace_size(ctypes.byref(d))
    ws = torch.empty((max(wsz, 4),), dtype=torch.uint8, device=dev)
    _check(_lib.hm_quantize_weight(ctypes.byref(d), _ptr(w), _ptr(zeros), _ptr(q), _ptr(scales), _ptr(g),
                                   _ptr(ws), wsz, _stream()), "hm_quantize_weight")
    return q, scales, g


def alloc_packed(d, device="cuda"):
    size = packed_size(d)
    if size == 0:
        raise HmError(1, "hm_packed_size")
    return torch.empty((size,), dtype=torch.uint8, device=device)


def transform(d, q, scales, zeros=None, out=None):
    _dev(("q", q), ("scales", scales), ("zeros", zeros), ("out", out))
    packed = alloc_packed(d, q.device) if out is None else out
    _check(_lib.hm_transform(ctypes.byref(d), _ptr(q), _ptr(scales), _ptr(zeros), _ptr(packed), _stream()),
           "hm_transform")
    return packed


def dequant(d, packed):
    _dev(("packed", packed))
    w = torch.empty((d.N, d.K), dtype=torch.bfloat16, device=packed.device)
    _check(_lib.hm_dequant(ctypes.byref(d), _ptr(packed), _ptr(w), _stream()), "hm_dequant")
    return w


def quant_act_fp8(x):
    _dev(("x", x))
    m, k = x.shape
    xq = torch.empty((m, k), dtype=torch.uint8, device=x.device)
    s = torch.empty((m,), dtype=torch.float32, device=x.device)
    _check(_lib.hm_quant_act_fp8(_ptr(x), m, k, _ptr(xq), _ptr(s), _stream()), "hm_quant_act_fp8")
    return xq, s


def silu_mul(gate_up, inter, out=None):
    """bf16 [rows][2*inter] (gate | up) -> bf16 SiLU(gate) * up [rows][inter] (hm_silu_mul)."""
    assert gate_up.dtype == torch.bfloat16 and gate_up.is_contiguous() and gate_up.shape[1] == 2 * inter
    rows = gate_up.shape[0]
    if out is None:
        out = torch.empty((rows, inter), dtype=torch.bfloat16, device=gate_up.device)
    assert out.dtype == torch.bfloat16 and out.is_contiguous() and tuple(out.shape) == (rows, inter)
    _check(_lib.hm_silu_mul(_ptr(gate_up), _ptr(out), int(rows), int(inter), _stream()), "hm_silu_mul")
    return out


def moe_gather(x, token_of_row, out=None):
    """bf16 x [T,K], int32 token_of_row [rows] (device) -> bf16 xs [rows,K] (hm_moe_gather)."""
    _dev(("x", x), ("token_of_row", token_of_row))
    if x.dtype != torch.bfloat16 or token_of_row.dtype != torch.int32:
        raise ValueError("x: bf16 [T,K]; token_of_row: int32 [rows]")
    t, k = x.shape
    rows = token_of_row.numel()
    xs = torch.empty((rows, k), dtype=torch.bfloat16, device=x.device) if out is None else _out(out, (rows, k))
    _check(_lib.hm_moe_gather(_ptr(x), _ptr(token_of_row), _ptr(xs), t, rows, k, _stream()), "hm_moe_gather")
    return xs


def moe_combine(y, pos, w, out=None):
    """bf16 y [rows,N], int32 pos [T,topk], fp32 w [T,topk] (device) -> bf16 [T,N] (hm_moe_combine)."""
    _dev(("y", y), ("pos", pos), ("w", w))
    if y.dtype != torch.bfloat16 or pos.dtype != torch.int32 or w.dtype != torch.float32 or pos.shape != w.shape:
        raise ValueError("y: bf16 [rows,N]; pos: int32 [T,topk]; w: float32 [T,topk]")
    rows, n = y.shape
    t, topk = pos.shape
    o = torch.empty((t, n), dtype=torch.bfloat16, device=y.device) if out is None else _out(out, (t, n))
    _check(_lib.hm_moe_combine(_ptr(y), _ptr(pos), _ptr(w), _ptr(o), t, topk, rows, n, _stream()),
           "hm_moe_combine")
    return o


def quant_act_nvfp4(x, g_in=None):
    _dev(("x", x), ("g_in", g_in))
    m, k = x.shape
    xq = torch.empty((m, k // 2), dtype=torch.uint8, device=x.device)
    xs = torch.empty((max(_lib.hm_act_scale_size(m, k), 1),), dtype=torch.uint8, device=x.device)
    g = torch.empty((1,), dtype=torch.float32, device=x.device)
    wsz = _lib.hm_act_workspace_size(m, k)
    ws = torch.empty((max(wsz, 4),), dtype=torch.uint8, device=x.device)
    _check(_lib.hm_quant_act_nvfp4(_ptr(x), m, k, _ptr(g_in), _ptr(xq), _ptr(xs), _ptr(g), _ptr(ws), wsz,
                                   _stream()), "hm_quant_act_nvfp4")
    return xq, xs, g


def workspace_size(fmt, m, n, k):
    return _lib.hm_workspace_size(int(fmt), int(m), int(n), int(k))


def alloc_workspace(fmt, m, n, k, device="cuda"):
    """Zero-filled workspace (the library needs its counters zero before first use)."""
    return torch.zeros((max(workspace_size(fmt, m, n, k), 256),), dtype=torch.uint8, device=device)


_WS_CACHE = {}


def cached_workspace(fmt, m, n, k, device, need=None):
    """A zero-initialised workspace kept per (device, current stream) and grown on demand, so that
    calls without `ws` allocate only when a problem needs more than any earlier one did (the
    library leaves its counters at zero after every call, so the buffer is reused as it is).
    Calls on one stream are ordered, so they may share it; other streams get their own.
    `need` (bytes) replaces the dense GEMM's size, e.g. hm_moe_workspace_size for the grouped GEMM."""
    need = max(workspace_size(fmt, m, n, k) if need is None else int(need), 256)
    key = (torch.device(device).index, torch.cuda.current_stream(device).cuda_stream)
    ws = _WS_CACHE.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros((need,), dtype=torch.uint8, device=device)
        _WS_CACHE[key] = ws
    return ws


def gemm(fmt, x, packed, n, k, x_scale=None, x_global=None, ws=None, out=None):
    _dev(("x", x), ("packed", packed), ("x_scale", x_scale), ("x_global", x_global), ("ws", ws))
    m = x.shape[0]
    y = torch.empty((m, n), dtype=torch.bfloat16, device=x.device) if out is None else _out(out, (m, n))
    if ws is None:
        ws = cached_workspace(fmt, m, n, k, x.device)
    _check(_lib.hm_gemm(int(fmt), _ptr(x), _ptr(x_scale), _ptr(x_global), _ptr(packed), _ptr(y), m, n, k,
                        _ptr(ws), ws.numel(), _stream()), "hm_gemm")
    return y


def gemm_noalloc(fmt, x, packed, n, k, out=None):
    """W4A16 GEMM through the allocation-free entry point (scratch inside the library)."""
    _dev(("x", x), ("packed", packed))
    m = x.shape[0]
    y = torch.empty((m, n), dtype=torch.bfloat16, device=x.device) if out is None else _out(out, (m, n))
    _check(_lib.hm_gemm_w4a16_noalloc(int(fmt), _ptr(x), _ptr(packed), _ptr(y), m, n, k, _stream()),
           "hm_gemm_w4a16_noalloc")
    return y


def moe_stride(d):
    """Bytes between experts in a strided MoE weight buffer: the packed size rounded up to 256."""
    return (packed_size(d) + 255) // 256 * 256


def alloc_moe_packed(d, experts, device="cuda"):
    """One buffer for `experts` packed weights of description d at moe_stride(d)."""
    return torch.empty((experts * moe_stride(d),), dtype=torch.uint8, device=device)


def moe_expert_view(buf, d, e):
    """Expert e's slot of a strided MoE weight buffer (to pass to transform(out=...))."""
    st = moe_stride(d)
    return buf[e * st:e * st + packed_size(d)]


def moe_gemm_strided(fmt, x, offsets, packed, experts, stride, n, k, x_scale=None, out=None, ws=None):
    """Grouped GEMM with the experts at packed + e * stride (hm_moe_gemm_strided). x: expert-sorted
    rows (bf16, or e4m3 bytes with x_scale for W4A8); offsets int32 [E+1] (device)."""
    _dev(("x", x), ("offsets", offsets), ("packed", packed), ("x_scale", x_scale), ("ws", ws))
    rows = x.shape[0]
    y = torch.empty((rows, n), dtype=torch.bfloat16, device=x.device) if out is None else _out(out, (rows, n))
    if ws is None:
        ws = cached_workspace(fmt, rows, n, k, x.device,
                              need=_lib.hm_moe_workspace_size(int(fmt), rows, int(experts), n, k))
    _check(_lib.hm_moe_gemm_strided(int(fmt), _ptr(x), _ptr(x_scale), _ptr(offsets), int(experts), _ptr(packed),
                                    int(stride), _ptr(y), rows, n, k, _ptr(ws), ws.numel(), _stream()),
           "hm_moe_gemm_strided")
    return y


def moe_gemm(fmt, x, offsets, packed_ptrs, n, k, out=None, ws=None):
    """x: expert-sorted rows [R,K] bf16; offsets int32 [E+1] (device); packed_ptrs int64 [E] (device).
    ws: a zero-initialised workspace of hm_moe_workspace_size bytes, by default the cached one."""
    _dev(("x", x), ("offsets", offsets), ("packed_ptrs", packed_ptrs), ("ws", ws))
    if offsets.dtype != torch.int32 or packed_ptrs.dtype != torch.int64 or packed_ptrs.numel() != offsets.numel() - 1:
        raise ValueError("offsets: int32 [E+1]; packed_ptrs: int64 [E]")
    rows = x.shape[0]
    e = offsets.numel() - 1
    y = torch.empty((rows, n), dtype=torch.bfloat16, device=x.device) if out is None else _out(out, (rows, n))
    if ws is None:
        ws = cached_workspace(fmt, rows, n, k, x.device, need=_lib.hm_moe_workspace_size(int(fmt), rows, e, n, k))
    _check(_lib.hm_moe_gemm(int(fmt), _ptr(x), _ptr(offsets), e, _ptr(packed_ptrs), _ptr(y), rows, n, k,
                            _ptr(ws), ws.numel(), _stream()), "hm_moe_gemm")
    return y


def plan(fmt, m, n, k, num_sms):
    info = PlanInfo()
    _check(_lib.hm_plan(int(fmt), int(m), int(n), int(k), int(num_sms), ctypes.byref(info)), "hm_plan")
    return {f: getattr(info, f) for f, _ in PlanInfo._fields_}


def device_error():
    """Returns and clears the device error word. A call that stopped early may leave arrival
    counters raised in its workspace, so a non-zero word also drops the cached workspaces."""
    v = int(_lib.hm_get_device_error(_stream()))
    if v:
        _WS_CACHE.clear()
    return v


def mma_peak(kind, iters, repeats=3):
    """Dense TFLOP/s of a tcgen05 MMA kind (0 f16, 1 mxf8f6f4, 2 mxf4nvf4) from hm_mma_peak_probe,
    timed with CUDA events on the current stream: the best of `repeats` launches after one warm-up."""
    fl = ctypes.c_double(0.0)
    _check(_lib.hm_mma_peak_probe(int(kind), int(iters), ctypes.byref(fl), _stream()), "hm_mma_peak_probe")
    best = None
    for _ in range(repeats):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        _check(_lib.hm_mma_peak_probe(int(kind), int(iters), ctypes.byref(fl), _stream()), "hm_mma_peak_probe")
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    return fl.value / (best * 1e-3) / 1e12, best


def debug_wait_timeout(ns):
    _check(_lib.hm_debug_wait_timeout(int(ns), _stream()), "hm_debug_wait_timeout")


def set_trace_buffer(buf):
    """Install a uint64 device tensor as the per-CTA timestamp buffer (None removes it)."""
    if buf is None:
        _check(_lib.hm_set_trace_buffer(None, 0), "hm_set_trace_buffer")
    else:
        _check(_lib.hm_set_trace_buffer(_ptr(buf), buf.numel() * buf.element_size()), "hm_set_trace_buffer")


def version():
    return _lib.hm_version().decode()
