#!/usr/bin/env python3
"""Throughput benchmark of the weight-quantized GEMM library on GB300.

Default workload: the W4A16 dense LLM-layer sweep -- (N, K) in {(4096, 4096), (14336, 4096),
(4096, 14336)} x M in {1, 2, 4, 8, 16, 32, 64, 128, 256, 1024, 4096, 8192}, INT4 weights with a
bf16 scale and a u4 zero-point (~U{0..15}) per 128 along K, X bf16 ~ N(0, 1), W ~ N(0, 0.02)
(seeded, generated on the device). Other workloads (--workload): w4a8 (MXFP4 x per-token FP8,
N=K=7168 and N=18432, K=7168), w4a4 (NVFP4, N=K=8192, M in {16, 128, 1024, 8192}), moe_w4a16 and
moe_mxfp4 (E=256 experts, gate-up N=4096/K=7168 and down N=7168/K=2048, top-8 Zipf(1.1) routing
of T in {16, 256, 4096, 16384} tokens).

A step runs every (shape, M) point of the workload once per rotation copy of its packed weight
(enough copies to cover 4x the L2 size, so every launch streams its weights from HBM); each
point is one CUDA graph of those launches. Per-point times come from CUDA events on the
launching stream. `value` is the aggregate TFLOP/s of the whole step; the per-point TFLOP/s,
weight GB/s and roofline fractions are in `sweep`. `e2e` repeats one pass over the points
through the public API with host (pinned) inputs and outputs, copies included: each point's input
is copied in on one stream, computed on the bench stream and its output copied back on a third, so
that the copies of neighbouring points overlap a point's compute (per point the order is copy in,
compute, copy out; a point's buffers are reused by the next pass only after its previous copy-out).

--impl reference times the CPU oracle (fp64 NumPy) on a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs an independent replica (the path does not shard);
rank 0 prints one JSON line.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantized GEMM TFLOP/s and weight GB/s vs M, % of GB300 HBM/tensor roofline"
MS = [1, 2, 4, 8, 16, 32, 64, 128, 256, 1024, 4096, 8192]
L2_BYTES = 126 * 1024 * 1024


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        pk = dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"], source="measured")
    else:
        pk = dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")
    kp = os.path.join(ROOT, "profiles", "tcgen05_peaks.json")
    if os.path.exists(kp):
        d = json.load(open(kp))
        pk["kinds"] = {k: v["tflops"] for k, v in d["kinds"].items()}
        pk["kinds_note"] = d.get("note", "")
    return pk


def measured_traffic(workload, label):
    """DRAM bytes per launch of the point's kernel from an ncu capture recorded under profiles/,
    or None when there is none or the kernel's sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    entry = json.load(open(path))["points"].get(f"{workload}:{label}")
    if entry is None:
        return None
    h = hashlib.sha256()
    for f in entry["sources"]:
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        h.update(open(fp, "rb").read())
    if h.hexdigest() != entry["sources_sha256"]:
        return None
    return entry["read_bytes"] + entry["write_bytes"]


# nominal dense ratios of the MMA kinds to kind::f16 (bf16) on GB300: 2.25 (bf16), 4.5 (fp8) and
# 13.5 (fp4) PFLOP/s dense, i.e. fp8 x2 and fp4 x6; used only when no measured peak of the kind
# is recorded (profiles/tcgen05_peaks.json, written from the tcgen05 microbenchmark)
KIND_RATIO = {"kind::f16": 1.0, "kind::mxf8f6f4": 2.0, "kind::mxf4nvf4": 6.0}


def tensor_peak(pk, kind):
    """Dense TFLOP/s of an MMA kind: the measured tcgen05 peak of that kind when recorded, else the
    measured cuBLAS bf16 figure times the nominal ratio."""
    kinds = pk.get("kinds") or {}
    if kind in kinds:
        return kinds[kind]
    return pk["bf16_sus"] * KIND_RATIO[kind]


def peak_source(pk, kind, bound):
    if bound != "tensor":
        return f"{pk['source']} (hbm copy)"
    if kind in (pk.get("kinds") or {}):
        return f"measured tcgen05 {kind} microbenchmark ({pk.get('kinds_note', '')})"
    extra = f" x nominal {KIND_RATIO[kind]} for {kind}" if kind != "kind::f16" else ""
    return f"{pk['source']} (bf16 sustained{extra})"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.path is None or not os.path.exists(self.path):
            return None
        sm, smax, reasons = [], [], set()
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                               f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- workloads

class Point:
    def __init__(self, label, fmt, m, n, k, flops, weight_bytes, act_bytes, out_bytes, kind, launches):
        self.label, self.fmt, self.m, self.n, self.k = label, fmt, m, n, k
        self.flops, self.weight_bytes, self.act_bytes, self.out_bytes = flops, weight_bytes, act_bytes, out_bytes
        self.kind, self.launches_per_call = kind, launches
        self.calls = []        # list of zero-arg callables, one per rotation copy
        self.reps = 1          # passes over the copies captured in the point's graph
        self.e2e = None        # (host_in, dev_in, host_out, dev_out, call)
        self.graph = None
        self.times_ms = []     # per launch, one value per timed step

    @property
    def launches(self):
        return self.reps * len(self.calls)

    @property
    def bytes(self):
        return self.weight_bytes + self.act_bytes + self.out_bytes


def rotations(weight_bytes):
    return max(2, math.ceil(4 * L2_BYTES / max(weight_bytes, 1)))


def dense_points(hm, synth, fmt, shapes, ms, seed0, kind, quick, has_zero=None):
    points = []
    for si, (n, k) in enumerate(shapes):
        if has_zero is None:
            has_zero = fmt == hm.W4A16_INT4
        d = hm.desc(fmt, n, k, has_zero)
        w = synth.device_weights(n, k, seed=seed0 + si)
        z = synth.device_zero_points(n, k // 128, seed=seed0 + 100 + si) if has_zero else None
        q, s, g = hm.quantize_weight(d, w, z)
        if fmt == hm.W4A4_NVFP4:
            d = hm.desc(fmt, n, k, False, float(g.item()))
        packed = hm.transform(d, q, s, z)
        del w, q, s
        payload = hm.packed_size(d) - 256
        copies = [packed] + [packed.clone() for _ in range(rotations(payload) - 1)]
        for m in ms:
            x = synth.device_activations(m, k, seed=seed0 + 1000 + m,
                                         outlier_frac=0.01 if fmt == hm.W4A8_MXFP4 else 0.0)
            y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
            ws = hm.alloc_workspace(fmt, m, n, k)
            if fmt in (hm.W4A16_INT4, hm.W4A16_MXFP4, hm.W4A16_MXINT4):
                act = 2 * m * k
                launches = 1
            elif fmt == hm.W4A8_MXFP4:
                act = 2 * m * k          # bf16 in, quantized inside the call
                launches = 2
            else:
                act = 2 * m * k
                launches = 3
            p = Point(f"{n}x{k} M={m}", fmt, m, n, k, 2.0 * m * n * k, payload, act, 2 * m * n, kind, launches)
            for c in copies:
                p.calls.append(lambda c=c, x=x, y=y, ws=ws, n=n, k=k, fmt=fmt: hm.gemm(fmt, x, c, n, k, ws=ws, out=y))
            xh = x.cpu().pin_memory()
            yh = torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
            p.e2e = (xh, x, yh, y, p.calls[0])
            points.append(p)
        torch.cuda.synchronize()
    if quick:
        points = [p for p in points if p.m in (1, 16, 1024)]
    return points


def moe_points(hm, synth, fmt, quick, only_t=None, experts=256, only_layer=None):
    """only_t: the T values to build instead of the default sweep (from --m); experts: E (256 in the
    benchmark, fewer for small profiling cases, --experts); only_layer: build one layer (--shape)."""
    e, topk = experts, 8
    layers = [(nm, n, k) for nm, n, k in (("gate_up", 4096, 7168), ("down", 7168, 2048))
              if only_layer in (None, "", nm)]
    tokens = only_t or ([16, 256, 4096, 16384] if not quick else [16, 4096])
    points = []
    for li, (name, n, k) in enumerate(layers):
        d = hm.desc(fmt, n, k, fmt == hm.W4A16_INT4)
        packs = []
        for ei in range(e):
            w = synth.device_weights(n, k, seed=10000 * (li + 1) + ei)
            z = synth.device_zero_points(n, k // 128, seed=20000 * (li + 1) + ei) if d.has_zero else None
            q, s, _ = hm.quantize_weight(d, w, z)
            packs.append(hm.transform(d, q, s, z))
            del w, q, s
        per_expert = hm.packed_size(d) - 256
        ptrs = torch.tensor([p.data_ptr() for p in packs], dtype=torch.int64, device="cuda")
        for t in tokens:
            _, _, offsets = synth.moe_routing(t, experts=e, topk=topk, seed=0)
            rows = int(offsets[-1])
            nonempty = int((np.diff(offsets) > 0).sum())
            x = synth.device_activations(rows, k, seed=30000 + t)
            y = torch.empty((rows, n), dtype=torch.bfloat16, device="cuda")
            offs = torch.from_numpy(offsets).cuda()
            p = Point(f"moe {name} T={t}", fmt, rows, n, k, 2.0 * rows * n * k, nonempty * per_expert,
                      2 * rows * k, 2 * rows * n, "kind::f16", 1)
            p.calls.append(lambda x=x, offs=offs, ptrs=ptrs, y=y, n=n, k=k: hm.moe_gemm(fmt, x, offs, ptrs, n, k, out=y))
            xh = x.cpu().pin_memory()
            yh = torch.empty((rows, n), dtype=torch.bfloat16).pin_memory()
            p.e2e = (xh, x, yh, y, p.calls[0])
            p._keep = (packs, ptrs)
            points.append(p)
        torch.cuda.synchronize()
    return points


def silu_points(hm, synth, quick):
    """MoE expert activation on the gate-up output of the MoE layers above: rows = 8 T,
    gate | up of 2 x 2048 columns in, 2048 out; inputs rotated over copies covering 4x L2."""
    inter = 2048
    tokens = [16, 256, 4096, 16384] if not quick else [16, 4096]
    points = []
    for t in tokens:
        rows = 8 * t
        gu = synth.device_activations(rows, 2 * inter, seed=40000 + t)
        h = torch.empty((rows, inter), dtype=torch.bfloat16, device="cuda")
        in_bytes, out_bytes = rows * 2 * inter * 2, rows * inter * 2
        # ~4 fp32 operations for SiLU and one multiply per output (no tensor-core work)
        p = Point(f"moe silu_mul T={t}", 0, rows, inter, 2 * inter, 5.0 * rows * inter, 0, in_bytes, out_bytes,
                  "kind::f16", 1)
        copies = [gu] + [gu.clone() for _ in range(rotations(in_bytes) - 1)]
        for c in copies:
            p.calls.append(lambda c=c, h=h: hm.silu_mul(c, inter, out=h))
        p.e2e = (gu.cpu().pin_memory(), gu, torch.empty((rows, inter), dtype=torch.bfloat16).pin_memory(), h,
                 p.calls[0])
        points.append(p)
    torch.cuda.synchronize()
    return points


def glue_points(hm, synth, quick):
    """MoE token gather (x[T, 7168] -> xs[8T, 7168] by the routing) and top-8 combine of the down
    layer's outputs (y[8T, 7168] -> out[T, 7168]) for the Zipf(1.1) routing of T tokens; inputs
    rotated over copies covering 4x L2. Bytes: the gather reads T x 7168 x 2 (every token row once)
    plus the row indices and writes 8T x 7168 x 2; the combine reads 8T x 7168 x 2 (+ routing) and
    writes T x 7168 x 2."""
    hidden, topk = 7168, 8
    tokens = [16, 256, 4096, 16384] if not quick else [16, 4096]
    points = []
    for t in tokens:
        tok, _, _, pos, wts = synth.moe_routing_slots(t, experts=256, topk=topk, seed=0)
        rows = t * topk
        x = synth.device_activations(t, hidden, seed=50000 + t)
        tok_d = torch.from_numpy(tok.astype(np.int32)).cuda()
        xs = torch.empty((rows, hidden), dtype=torch.bfloat16, device="cuda")
        # each token row is read from HBM once (its other copies come from L2) and written top-k times
        p = Point(f"moe gather T={t}", 0, rows, hidden, hidden, 0.0, 0, t * hidden * 2 + rows * 4, rows * hidden * 2,
                  "kind::f16", 1)
        copies = [x] + [x.clone() for _ in range(rotations(t * hidden * 2) - 1)]
        for c in copies:
            p.calls.append(lambda c=c, xs=xs, tok_d=tok_d: hm.moe_gather(c, tok_d, out=xs))
        p.e2e = (x.cpu().pin_memory(), x, torch.empty((rows, hidden), dtype=torch.bfloat16).pin_memory(), xs,
                 p.calls[0])
        points.append(p)
        y = synth.device_activations(rows, hidden, seed=60000 + t)
        pos_d = torch.from_numpy(pos.astype(np.int32)).cuda()
        w_d = torch.from_numpy(wts).cuda()
        out = torch.empty((t, hidden), dtype=torch.bfloat16, device="cuda")
        c_in = rows * hidden * 2 + t * topk * 8
        # one multiply-add per slot and output element
        p = Point(f"moe combine T={t}", 0, t, hidden, topk, 2.0 * t * topk * hidden, 0, c_in, t * hidden * 2,
                  "kind::f16", 1)
        copies = [y] + [y.clone() for _ in range(rotations(rows * hidden * 2) - 1)]
        for c in copies:
            p.calls.append(lambda c=c, out=out, pos_d=pos_d, w_d=w_d: hm.moe_combine(c, pos_d, w_d, out=out))
        p.e2e = (y.cpu().pin_memory(), y, torch.empty((t, hidden), dtype=torch.bfloat16).pin_memory(), out,
                 p.calls[0])
        points.append(p)
    torch.cuda.synchronize()
    return points


def build_points(args, hm, synth):
    pts = _build_points(args, hm, synth)
    if args.m:
        keep = {int(v) for v in args.m.split(",")}
        pts = [p for p in pts if p.m in keep or any(p.label.endswith(f"T={v}") for v in keep)]
    if args.shape:
        pts = [p for p in pts if p.label.startswith(args.shape + " ") or f" {args.shape} " in p.label]
    if not pts:
        raise SystemExit("no benchmark point matches the filters")
    return pts


def moe_ts(args):
    return sorted({int(v) for v in args.m.split(",")}) if args.m else None


def _build_points(args, hm, synth):
    w = args.workload
    if w == "w4a16":
        return dense_points(hm, synth, hm.W4A16_INT4, [(4096, 4096), (14336, 4096), (4096, 14336)], MS, 1,
                            "kind::f16", args.quick)
    if w == "w4a8":
        return dense_points(hm, synth, hm.W4A8_MXFP4, [(7168, 7168), (18432, 7168)], MS, 2, "kind::mxf8f6f4",
                            args.quick)
    if w == "w4a4":
        return dense_points(hm, synth, hm.W4A4_NVFP4, [(8192, 8192)], [16, 128, 1024, 8192], 3, "kind::mxf4nvf4",
                            args.quick)
    if w == "moe_w4a16":
        return moe_points(hm, synth, hm.W4A16_INT4, args.quick, moe_ts(args), args.experts, args.shape)
    if w == "moe_mxfp4":
        return moe_points(hm, synth, hm.W4A16_MXFP4, args.quick, moe_ts(args), args.experts, args.shape)
    if w == "w4a16_mxint4":
        return dense_points(hm, synth, hm.W4A16_MXINT4, [(4096, 4096), (14336, 4096), (4096, 14336)], MS, 4,
                            "kind::f16", args.quick)
    if w == "moe_mxint4":
        return moe_points(hm, synth, hm.W4A16_MXINT4, args.quick, moe_ts(args), args.experts, args.shape)
    if w == "moe_silu_mul":
        return silu_points(hm, synth, args.quick)
    if w == "moe_glue":
        return glue_points(hm, synth, args.quick)
    if w == "w4a16_tiny":
        return dense_points(hm, synth, hm.W4A16_INT4, [(256, 512)], [4], 0, "kind::f16", False, has_zero=False)
    raise SystemExit(f"unknown workload {w}")


EXTRA_WORKLOADS = ["w4a16_tiny", "w4a8", "w4a4", "moe_w4a16", "moe_mxfp4", "w4a16_mxint4", "moe_mxint4",
                   "moe_silu_mul", "moe_glue"]
DTYPE = {"w4a8": "fp8xfp4", "w4a4": "fp4"}
L2_NOTE = {"moe_silu_mul": "gate-up inputs rotated over copies covering 4x L2",
           "moe_glue": "token activations / expert outputs rotated over copies covering 4x L2",
           "w4a16_tiny": "packed weight rotated over copies covering 4x L2"}

WORKLOAD_NAMES = {
    "w4a16": "W4A16 dense LLM layer: (N,K) in {(4096,4096),(14336,4096),(4096,14336)} x M in "
             "{1,2,4,8,16,32,64,128,256,1024,4096,8192}; INT4 g128 bf16 scales + u4 zero-points",
    "w4a8": "W4A8-MXFP4 dense: (N,K) in {(7168,7168),(18432,7168)} x M sweep 1..8192; e2m1 + E8M0/32, "
            "per-token FP8 e4m3 activations (1% outliers x10) quantized inside the call",
    "w4a4": "W4A4-NVFP4 dense: N=K=8192, M in {16,128,1024,8192}; activations quantized inside the call",
    "moe_w4a16": "MoE grouped W4A16 INT4: E=256, gate-up 4096x7168 and down 7168x2048, top-8 Zipf(1.1), "
                 "T in {16,256,4096,16384}",
    "moe_mxfp4": "MoE grouped MXFP4-W4A16: E=256, gate-up 4096x7168 and down 7168x2048, top-8 Zipf(1.1), "
                 "T in {16,256,4096,16384}",
    "w4a16_mxint4": "MXINT4-W4A16 dense LLM layer: (N,K) in {(4096,4096),(14336,4096),(4096,14336)} x M in "
                    "{1,2,4,8,16,32,64,128,256,1024,4096,8192}; signed int4 + E8M0 scale per 32",
    "moe_mxint4": "MoE grouped MXINT4-W4A16: E=256, gate-up 4096x7168 and down 7168x2048, top-8 Zipf(1.1), "
                  "T in {16,256,4096,16384}",
    "w4a16_tiny": "W4A16 dense tiny: M=4, K=512, N=256, INT4 symmetric g128 bf16 scales",
    "moe_glue": "MoE token gather (T x 7168 -> 8T rows) and top-8 weighted combine (8T x 7168 -> T rows), "
                "Zipf(1.1) routing over 256 experts, T in {16,256,4096,16384} (HBM-bound; roofline in GB/s)",
    "moe_silu_mul": "MoE expert activation h = SiLU(gate) * up between the grouped GEMMs: rows = 8 T, "
                    "gate | up 2 x 2048 bf16 in, 2048 bf16 out, T in {16,256,4096,16384} (HBM-bound; "
                    "value in TFLOP/s of ~5 operations per output, roofline in GB/s)",
}


# ----------------------------------------------------------------------------- our arm

MIN_LAUNCHES = 200          # launches per point and timed step (CUDA graph of back-to-back calls)
SLOW_LAUNCH_MS = 0.5        # points slower than this per launch: >= 20 launches and >= 100 ms per step


def set_reps(points, stream):
    """Passes over the rotation copies per graph: at least MIN_LAUNCHES launches, or for slow
    points (> SLOW_LAUNCH_MS per launch, from one timed warm-up pass) at least 20 launches and
    100 ms."""
    for p in points:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for c in p.calls:
            c()
        b.record(stream)
        torch.cuda.synchronize()
        per = a.elapsed_time(b) / len(p.calls)
        want = MIN_LAUNCHES if per <= SLOW_LAUNCH_MS else max(20, math.ceil(100.0 / per))
        p.reps = max(1, math.ceil(want / len(p.calls)))


def measure(points, steps, warmup, stream, hm, world=1, clocks_index=None):
    """Capture one graph per point (reps x copies launches), replay each once per step; returns
    (total ms of the timed steps, clocks summary). Per-launch times per step land in p.times_ms."""
    for p in points:
        for c in p.calls:
            c()
    torch.cuda.synchronize()
    set_reps(points, stream)
    for p in points:
        p.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(p.graph, stream=stream):
            for _ in range(p.reps):
                for c in p.calls:
                    c()
    torch.cuda.synchronize()
    if hm.device_error() != 0:
        raise SystemExit("device error during warm-up")

    def step(events=None):
        for i, p in enumerate(points):
            if events is not None:
                events[i][0].record(stream)
            p.graph.replay()
            if events is not None:
                events[i][1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in points] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clk = Clocks(clocks_index) if clocks_index is not None else None
    if clk is not None:
        clk.__enter__()
    try:
        t0.record(stream)
        for s in range(steps):
            step(evs[s])
        t1.record(stream)
        torch.cuda.synchronize()
    finally:
        if clk is not None:
            clk.__exit__()
    barrier(world)
    for s in range(steps):
        for i, p in enumerate(points):
            p.times_ms.append(evs[s][i][0].elapsed_time(evs[s][i][1]) / p.launches)
    return t0.elapsed_time(t1), (clk.summary() if clk is not None else None)


def summarize(points, pk, workload, hm, local_rank):
    """Per-point sweep (median over the timed steps of the per-launch time) and the roofline of
    the point that takes the largest share of the step."""
    sweep = []
    dom, dom_share = None, -1.0
    total_pt = sum(statistics.median(p.times_ms) * p.launches for p in points)
    sms = torch.cuda.get_device_properties(local_rank).multi_processor_count
    for p in points:
        t = statistics.median(p.times_ms) * 1e-3
        peak_t = tensor_peak(pk, p.kind)
        tf = p.flops / t / 1e12
        gbs = p.bytes / t / 1e9
        share = t * 1e3 * p.launches / total_pt
        bound = "hbm" if (p.flops == 0 or p.bytes / (pk["hbm"] * 1e9) > p.flops / (peak_t * 1e12)) else "tensor"
        plan = None
        if p.fmt and not p.label.startswith("moe"):
            plan = hm.plan(p.fmt, p.m, p.n, p.k, sms)
            plan = {k: plan[k] for k in ("kernel", "tile_m", "stages", "stream_k", "grid")}
        sweep.append({"point": p.label, "plan": plan, "us": round(t * 1e6, 2), "launches": p.launches,
                      "tflops": round(tf, 2), "gbs": round(gbs, 1),
                      "weight_gbs": round(p.weight_bytes / t / 1e9, 1), "bound": bound,
                      "frac_hbm": round(gbs / pk["hbm"], 3), "frac_tensor": round(tf / peak_t, 3),
                      "share": round(share, 4)})
        if share > dom_share:
            dom, dom_share = p, share
    t = statistics.median(dom.times_ms) * 1e-3
    peak_t = tensor_peak(pk, dom.kind)
    dom_bound = "hbm" if (dom.flops == 0 or dom.bytes / (pk["hbm"] * 1e9) > dom.flops / (peak_t * 1e12)) else "tensor"
    if dom_bound == "tensor":
        ach, peak, unit = dom.flops / t / 1e12, peak_t, "TFLOP/s"
    else:
        ach, peak, unit = dom.bytes / t / 1e9, pk["hbm"], "GB/s"
    roofline = {"bound": dom_bound, "achieved": round(ach, 2), "peak": peak, "unit": unit,
                "frac": round(ach / peak, 4), "traffic": measured_traffic(workload, dom.label), "kernel": dom.label,
                "peak_source": peak_source(pk, dom.kind, dom_bound)}
    one = (pk.get("kinds") or {}).get(ONE_ISSUER_F16)
    if dom_bound == "tensor" and dom.kind == "kind::f16" and one:
        # what one issuing thread sustains with the 256-token tile's instruction (probe kind 5)
        roofline["one_issuer_ceiling"] = {"value": one, "frac": round(ach / one, 4), "source": ONE_ISSUER_F16}
    return sweep, roofline


KIND_PROBES = {"kind::f16": (0,), "kind::mxf8f6f4": (1, 3), "kind::mxf4nvf4": (2, 4)}
ONE_ISSUER_F16 = "kind::f16 M=128 N=256, A in TMEM, one issuing thread"


def live_kind_peaks(hm):
    """Dense TFLOP/s of each tcgen05 MMA kind on this device, from the library's throughput probe
    (the larger of its shapes per kind), or None when the probe fails."""
    try:
        out = {}
        for kind, probes in KIND_PROBES.items():
            out[kind] = round(max(hm.mma_peak(k, 20000 if k != 2 else 40000, repeats=3)[0] for k in probes), 1)
        # context, not a denominator: the W4A16 256-token tile's instruction from one issuing thread
        out[ONE_ISSUER_F16] = round(hm.mma_peak(5, 20000, repeats=3)[0], 1)
        if hm.device_error() != 0:
            return None
        return out
    except Exception:   # noqa: BLE001 - fall back to the recorded peaks
        return None


def run_ours(args, rank, world, local_rank):
    torch.cuda.set_device(local_rank)
    from moe_hm_gemm_gb300 import hm, synth
    pk = peaks()
    if not args.no_peak_probe:
        live = live_kind_peaks(hm)
        if live is not None:
            pk["kinds"] = live
            pk["kinds_note"] = "measured in this run by hm_mma_peak_probe"
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        points = build_points(args, hm, synth)
        total_ms, clocks = measure(points, args.steps, args.warmup, stream, hm, world, local_rank)
        err = hm.device_error()

        # end-to-end pass through the public API with host buffers
        e2e_ms = None
        h2d = d2h = 0
        if not args.no_e2e:
            s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
            last_out = {}      # point index -> event after its last copy-out (buffers free again)

            def e2e_pass():
                for i, p in enumerate(points):
                    xh, xd, yh, yd, call = p.e2e
                    with torch.cuda.stream(s_in):
                        if i in last_out:
                            s_in.wait_event(last_out[i])
                        xd.copy_(xh, non_blocking=True)
                        ready = torch.cuda.Event()
                        ready.record(s_in)
                    with torch.cuda.stream(stream):
                        stream.wait_event(ready)
                        call()
                        done = torch.cuda.Event()
                        done.record(stream)
                    with torch.cuda.stream(s_out):
                        s_out.wait_event(done)
                        yh.copy_(yd, non_blocking=True)
                        out = torch.cuda.Event()
                        out.record(s_out)
                    last_out[i] = out

            e2e_pass()
            torch.cuda.synchronize()
            reps = max(1, args.steps)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            s_in.wait_event(a)
            s_out.wait_event(a)
            for _ in range(reps):
                e2e_pass()
            for s_ in (s_in, s_out):
                tail = torch.cuda.Event()
                tail.record(s_)
                stream.wait_event(tail)
            b.record(stream)
            torch.cuda.synchronize()
            e2e_ms = a.elapsed_time(b) / reps
            h2d = sum(p.e2e[0].numel() * p.e2e[0].element_size() for p in points)
            d2h = sum(p.e2e[2].numel() * p.e2e[2].element_size() for p in points)
        sweep, roofline = summarize(points, pk, args.workload, hm, local_rank)
        flops_step = sum(p.flops * p.launches for p in points)
        flops_e2e_pass = sum(p.flops for p in points)
        launches = args.steps * sum(p.launches_per_call * p.launches for p in points)
        for p in points:
            p.graph = None
        del points
        torch.cuda.empty_cache()

        # the other configurations, each measured the same way and reported under "configs"
        configs = {}
        if not args.no_extra and args.workload == "w4a16" and not args.m and not args.shape:
            for w in EXTRA_WORKLOADS:
                sub = argparse.Namespace(**vars(args))
                sub.workload, sub.quick = w, False
                pts = _build_points(sub, hm, synth)
                ms_total, _ = measure(pts, args.extra_steps, 2, stream, hm, world)
                sw, rf = summarize(pts, pk, w, hm, local_rank)
                fl = sum(p.flops * p.launches for p in pts)
                configs[w] = {"workload": WORKLOAD_NAMES[w], "value": round(fl / (ms_total / args.extra_steps * 1e-3) / 1e12, 3),
                              "unit": "TFLOP/s", "steps": args.extra_steps, "roofline": rf, "sweep": sw}
                launches += args.extra_steps * sum(p.launches_per_call * p.launches for p in pts)
                for p in pts:
                    p.graph = None
                del pts
                torch.cuda.empty_cache()
            err |= hm.device_error()

    step_ms = total_ms / args.steps
    value, step_ms_max = aggregate_tflops(flops_step, step_ms, world)
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE.get(args.workload, "bf16"),
        "data": "synthetic (seeded, generated on the device)",
        "config": {"workload": WORKLOAD_NAMES[args.workload], "parallelism": f"replicas x{world}",
                   "l2": L2_NOTE.get(args.workload, "packed weights rotated over copies covering 4x L2 per shape"),
                   "timing": f"per point: one CUDA graph of >= {MIN_LAUNCHES} back-to-back launches "
                             f"(>= 20 launches and >= 100 ms for launches above {SLOW_LAUNCH_MS} ms), replayed once "
                             f"per step; per-point time = median over the timed steps"},
        "roofline": roofline, "gpu_launches": launches, "clocks": clocks, "device_error": err,
        "peaks": {"hbm_gbs": pk["hbm"], "bf16_tflops": pk["bf16"], "bf16_tflops_sustained": pk["bf16_sus"],
                  "tensor_kind_tflops": pk.get("kinds"), "source": pk["source"]},
        "sweep": sweep,
    }
    if configs:
        out["configs"] = configs
    if e2e_ms is not None:
        out["e2e"] = {"value": round(world * flops_e2e_pass / (max_over_ranks(e2e_ms, world) * 1e-3) / 1e12, 3),
                      "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if rank == 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(args.workload, seconds=args.cpu_seconds)
        print(json.dumps(out), flush=True)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v, world, device="cuda"):
    """The slowest rank's time: replicas run concurrently, so the job ends with the last one."""
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(work_flops_per_rank, ms_per_step, world, device="cuda"):
    """Whole-job throughput of N replicas: all ranks' work over the max-over-ranks step time."""
    ms = max_over_ranks(ms_per_step, world, device)
    return world * work_flops_per_rank / (ms * 1e-3) / 1e12, ms


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(workload):
    """A bounded sample of the workload for the CPU oracle: (description, flops, run callable)."""
    from moe_hm_gemm_gb300 import synth
    from oracle import gemm as og
    from oracle import quant as oq
    if workload in ("w4a16_mxint4", "moe_mxint4", "moe_mxfp4"):
        n, k, m = 4096, 4096, 64
        w = synth.weights(n, k, seed=1)
        x = synth.activations(m, k, seed=3).float().numpy().astype(np.float64)
        if workload == "moe_mxfp4":
            codes, e = oq.quant_mxfp4(w)
            return (f"oracle MXFP4-W4A16 dequant + fp64 GEMM, N=K=4096, M={m} rows", 2.0 * m * n * k,
                    lambda: og.gemm_w4a16_mxfp4(x, codes, e))
        q, e = oq.quant_mxint4(w)
        return (f"oracle MXINT4-W4A16 dequant + fp64 GEMM, N=K=4096, M={m} rows", 2.0 * m * n * k,
                lambda: og.gemm_w4a16_mxint4(x, q, e))
    if workload in ("w4a16", "moe_w4a16"):
        n, k, m = 4096, 4096, 64
        w = synth.weights(n, k, seed=1)
        z = synth.zero_points(n, k // 128, seed=2)
        q, s = oq.quant_int4(w, zeros=z)
        x = synth.activations(m, k, seed=3).float().numpy().astype(np.float64)
        desc = f"oracle W4A16 INT4+zp dequant + fp64 GEMM, N=K=4096, M={m} rows"
        return desc, 2.0 * m * n * k, lambda: og.gemm_w4a16_int4(x, q, s, z)
    if workload == "w4a16_tiny":
        n, k, m = 256, 512, 4
        q, s_ = oq.quant_int4(synth.weights(n, k, seed=0))
        x = synth.activations(m, k, seed=0).float().numpy().astype(np.float64)
        return (f"oracle W4A16 INT4 dequant + fp64 GEMM, N=256, K=512, M={m}", 2.0 * m * n * k,
                lambda: og.gemm_w4a16_int4(x, q, s_))
    if workload == "moe_glue":
        from oracle import moe as om
        t, hidden = 256, 7168
        tok, _, _, pos, wts = synth.moe_routing_slots(t, experts=256, topk=8, seed=0)
        x = synth.activations(t, hidden, seed=1).float().numpy().astype(np.float64)
        y = synth.activations(8 * t, hidden, seed=2).float().numpy().astype(np.float64)
        return (f"oracle MoE gather + top-8 combine in fp64, T={t}, hidden {hidden}", 2.0 * t * 8 * hidden,
                lambda: (om.gather_rows(x, tok), om.combine(y, pos, wts)))
    if workload == "moe_silu_mul":
        from oracle import act as oa
        rows, inter = 4096, 2048
        gu = synth.activations(rows, 2 * inter, seed=3).float().numpy().astype(np.float64)
        return (f"oracle SiLU(gate) * up in fp64 + bf16 rounding, {rows} rows x {inter}", 5.0 * rows * inter,
                lambda: oa.silu_mul(gu, inter))
    if workload == "w4a8":
        n, k, m = 7168, 7168, 64
        codes, e = oq.quant_mxfp4(synth.weights(n, k, seed=1))
        x = synth.activations(m, k, seed=3, outlier_frac=0.01).float().numpy().astype(np.float64)

        def run():
            xq, st = oq.quant_fp8_per_token(x)
            return og.gemm_w4a8_mxfp4(xq, st, codes, e)
        return f"oracle W4A8 FP8 act-quant + dequant + fp64 GEMM, N=K=7168, M={m}", 2.0 * m * n * k, run
    n, k, m = 8192, 8192, 16
    wc, wsb, gw = oq.quant_nvfp4(synth.weights(n, k, seed=1))
    x = synth.activations(m, k, seed=3).float().numpy().astype(np.float64)

    def run():
        xc, xsb, gx = oq.quant_nvfp4(x)
        return og.gemm_w4a4_nvfp4(xc, xsb, gx, wc, wsb, gw)
    return f"oracle W4A4 NVFP4 act-quant + dequant + fp64 GEMM, N=K=8192, M={m}", 2.0 * m * n * k, run


def cpu_baseline(workload, seconds=15.0):
    desc, flops, run = oracle_sample(workload)
    run()
    t0 = time.perf_counter()
    reps = 0
    while time.perf_counter() - t0 < seconds:
        run()
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{desc}; {reps} repetitions, {dt:.2f} s each"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    desc, flops, run = oracle_sample(args.workload)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = flops / dt / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
           "config": {"workload": WORKLOAD_NAMES[args.workload], "sample": desc},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                            "sample": desc},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_NAMES), default="w4a16")
    ap.add_argument("--quick", action="store_true", help="a subset of M values (for profiling)")
    ap.add_argument("--m", default="", help="comma-separated M (or MoE T) values to keep")
    ap.add_argument("--shape", default="", help="keep one NxK shape, e.g. 4096x4096 (MoE: gate_up/down)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--experts", type=int, default=256,
                    help="MoE workloads: experts E (the benchmark's 256; fewer for small profiling cases)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads the default run reports under 'configs'")
    ap.add_argument("--extra-steps", type=int, default=5)
    ap.add_argument("--no-peak-probe", action="store_true",
                    help="take the MMA-kind peaks from profiles/tcgen05_peaks.json instead of measuring them")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
