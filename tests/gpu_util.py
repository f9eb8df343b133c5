"""Helpers shared by the GPU tests: standard-format tensors from the oracle's quantizers,
oracle references, and the tolerance check. Test infrastructure only."""
import numpy as np
import torch

from oracle import gemm as og
from oracle import layout as ol
from oracle import quant as oq


def pack_nibbles(codes):
    """[R,K] codes 0..15 (or signed INT4) -> uint8 [R,K/2], even k in the low nibble."""
    c = (np.asarray(codes) & 0xF).astype(np.uint8)
    return c[:, 0::2] | (c[:, 1::2] << 4)


def to_bf16(values):
    """bf16-exact float64 values -> torch bf16 (the conversion is exact)."""
    return torch.from_numpy(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)


class QuantWeight:
    """A weight quantized by the oracle, with its standard-format tensors."""

    def __init__(self, fmt, w, zeros=None, group=0):
        self.fmt = fmt
        self.n, self.k = w.shape
        self.zeros = zeros
        self.g = 1.0
        self.group = group
        if fmt == ol.FMT_W4A16_INT4:
            grp = self.k if group == -1 else (group or 128)
            self.q, self.s = oq.quant_int4(w, zeros=zeros, group=grp)
            self.what = oq.dequant_int4(self.q, self.s, zeros, group=grp)
            self.std_q = pack_nibbles(self.q)
            self.std_s = to_bf16(self.s)
            self.packed_ref = ol.pack_w4a16_int4(self.q, self.s, zeros, group=grp)
        elif fmt == ol.FMT_W4A16_INT4_G32:
            grp = group or 32
            self.q, self.s = oq.quant_int4(w, zeros=zeros, group=grp)
            self.what = oq.dequant_int4(self.q, self.s, zeros, group=grp)
            self.std_q = pack_nibbles(self.q)
            self.std_s = to_bf16(self.s)
            self.packed_ref = ol.pack_w4a16_int4_g32(self.q, self.s, zeros, group=grp)
        elif fmt == ol.FMT_W8A16_INT8:
            self.q, self.s = oq.quant_int8(w, zeros=zeros)
            self.what = oq.dequant_int8(self.q, self.s, zeros)
            self.std_q = (np.asarray(self.q) & 0xFF).astype(np.uint8)      # one byte per code
            self.std_s = to_bf16(self.s)
            self.packed_ref = ol.pack_w8a16_int8(self.q, self.s, zeros)
        elif fmt in (ol.FMT_W4A16_MXFP4, ol.FMT_W4A8_MXFP4):
            self.q, self.s = oq.quant_mxfp4(w)
            self.what = oq.dequant_mxfp4(self.q, self.s)
            self.std_q = pack_nibbles(self.q)
            self.std_s = torch.from_numpy(self.s.astype(np.uint8))
            pack = ol.pack_w4a16_mxfp4 if fmt == ol.FMT_W4A16_MXFP4 else ol.pack_w4a8_mxfp4
            self.packed_ref = pack(self.q, self.s)
        elif fmt == ol.FMT_W4A16_MXINT4:
            self.q, self.s = oq.quant_mxint4(w)
            self.what = oq.dequant_mxint4(self.q, self.s)
            self.std_q = pack_nibbles(self.q)            # two's-complement nibbles
            self.std_s = torch.from_numpy(self.s.astype(np.uint8))
            self.packed_ref = ol.pack_w4a16_mxint4(self.q, self.s)
        else:
            self.q, self.s, self.g = oq.quant_nvfp4(w)
            self.what = oq.dequant_nvfp4(self.q, self.s, self.g)
            self.std_q = pack_nibbles(self.q)
            self.std_s = torch.from_numpy(self.s.astype(np.uint8))
            self.packed_ref = ol.pack_w4a4_nvfp4(self.q, self.s, self.g)

    def device_inputs(self):
        z = None if self.zeros is None else torch.from_numpy(np.asarray(self.zeros, np.uint8)).cuda()
        return torch.from_numpy(self.std_q).cuda(), self.std_s.cuda(), z

    def desc(self, hm, zero_convention=0):
        return hm.desc(self.fmt, self.n, self.k, self.zeros is not None, self.g, group=self.group,
                       zero_convention=zero_convention)

    def transform(self, hm):
        d = self.desc(hm)
        q, s, z = self.device_inputs()
        return d, hm.transform(d, q, s, z)


CANARY = -3.0
CANARY_ROWS = 3


def canary_out(m, n):
    """An output of m bf16 rows followed by CANARY_ROWS rows of CANARY in one buffer; returns
    (buffer, its first m rows). A kernel that stores past row m - 1 overwrites the canary."""
    full = torch.full((m + CANARY_ROWS, n), CANARY, dtype=torch.bfloat16, device="cuda")
    return full, full[:m]


def check_canary(full, m, what=""):
    assert bool((full[m:] == CANARY).all()), f"{what}: a kernel wrote past the {m} output rows"


def assert_close(y_gpu, yref, what=""):
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    ok = og.tolerance_ok(y, yref)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        details = [(tuple(i), y[tuple(i)], yref[tuple(i)]) for i in bad]
        raise AssertionError(f"{what}: {int((~ok).sum())}/{ok.size} outside tolerance, e.g. {details}")


def bf16_np(t):
    return t.float().cpu().numpy().astype(np.float64)
