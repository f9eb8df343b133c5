"""Seeded synthetic inputs shaped like the weight-quantized GEMM workloads.

This module only draws random numbers; it holds none of the method's arithmetic (no
quantization, packing or GEMM). Both the CUDA path (tests, bench) and the CPU oracle
(tests) take their inputs from here.

Recipes (shapes and distributions of the LLM-layer and MoE workloads):
  * weights W[N,K] fp32 ~ N(0, 0.02);
  * activations X[M,K] ~ N(0, 1) stored as bf16, optionally with a fraction of entries
    (uniform positions) multiplied by 10 ("outliers");
  * zero-points u4 ~ U{0..15} per (row, group of 128);
  * MoE routing: each token picks top-k distinct experts with p_i proportional to
    i^-alpha (Zipf, alpha = 1.1) over E experts; rows are the (token, expert) pairs
    sorted stably by expert, with int32 offsets[E+1].

CPU generators use numpy's default_rng(seed); the large-shape generators used by the
benchmark draw on the GPU with a seeded torch generator.
"""
import numpy as np
import torch


def weights(n, k, seed, std=0.02):
    return (np.random.default_rng(seed).standard_normal((n, k), dtype=np.float32) * np.float32(std))


def activations(m, k, seed, outlier_frac=0.0, outlier_scale=10.0):
    """bf16 tensor [m,k] (CPU)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k), dtype=np.float32)
    if outlier_frac > 0 and x.size:
        cnt = int(round(outlier_frac * x.size))
        idx = rng.choice(x.size, size=cnt, replace=False)
        x.reshape(-1)[idx] *= np.float32(outlier_scale)
    return torch.from_numpy(x).to(torch.bfloat16)


def zero_points(n, groups, seed):
    return np.random.default_rng(seed).integers(0, 16, size=(n, groups), dtype=np.uint8)


def moe_routing(tokens, experts=256, topk=8, alpha=1.1, seed=0):
    """Returns (token_of_row int64 [T*topk], expert_of_row int64 [T*topk], offsets int32 [E+1])."""
    rng = np.random.default_rng(seed)
    p = np.arange(1, experts + 1, dtype=np.float64) ** (-alpha)
    p /= p.sum()
    choice = np.stack([rng.choice(experts, topk, replace=False, p=p) for _ in range(tokens)]) \
        if tokens else np.zeros((0, topk), dtype=np.int64)
    tok = np.repeat(np.arange(tokens), topk)
    exp = choice.reshape(-1).astype(np.int64)
    order = np.argsort(exp, kind="stable")
    counts = np.bincount(exp, minlength=experts)
    offsets = np.zeros(experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return tok[order], exp[order], offsets


def moe_routing_slots(tokens, experts=256, topk=8, alpha=1.1, seed=0):
    """moe_routing plus, for the combine after the grouped GEMMs, pos [T][topk] int32 (the sorted row
    holding token t's j-th routing choice) and weights [T][topk] float32 (a softmax of N(0,1) logits
    per token)."""
    rng = np.random.default_rng(seed)
    p = np.arange(1, experts + 1, dtype=np.float64) ** (-alpha)
    p /= p.sum()
    choice = np.stack([rng.choice(experts, topk, replace=False, p=p) for _ in range(tokens)]) \
        if tokens else np.zeros((0, topk), dtype=np.int64)
    tok = np.repeat(np.arange(tokens), topk)
    exp = choice.reshape(-1).astype(np.int64)
    order = np.argsort(exp, kind="stable")
    counts = np.bincount(exp, minlength=experts)
    offsets = np.zeros(experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    pos = np.empty(tokens * topk, dtype=np.int32)
    pos[order] = np.arange(tokens * topk, dtype=np.int32)
    logits = rng.standard_normal((tokens, topk))
    wts = np.exp(logits - logits.max(axis=1, keepdims=True)) if tokens else logits
    wts = (wts / wts.sum(axis=1, keepdims=True)).astype(np.float32) if tokens else wts.astype(np.float32)
    return tok[order], exp[order], offsets, pos.reshape(tokens, topk), wts


def device_weights(n, k, seed, device="cuda", std=0.02):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * std


def device_activations(m, k, seed, device="cuda", outlier_frac=0.0, outlier_scale=10.0):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0 and x.numel():
        mask = torch.rand((m, k), generator=g, device=device) < outlier_frac
        x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def device_zero_points(n, groups, seed, device="cuda"):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(0, 16, (n, groups), generator=g, device=device, dtype=torch.uint8)
