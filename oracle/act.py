"""The MoE expert activation between the two grouped GEMMs, in fp64 (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU baseline use this module; the product
path never does.

The MoE layer the pages measure (the explainer page "vLLM Humming은 4비트를 어떻게 계산하나",
MoE paragraph of the section "같은 가중치도 한 토큰과 많은 토큰에서 비용이 다르다", and the
DeepSeek end-to-end runs on the news pages, section "하나의 라이브러리로 긴 포맷 목록을 포괄")
runs each expert's gate-up GEMM, an activation, then its down GEMM. The pages do not print the
activation; the reading taken here is the gated SiLU of such expert MLPs:
    h = SiLU(gate) * up,   SiLU(v) = v / (1 + exp(-v)),
with gate the first half and up the second half of each gate-up output row, and h rounded once
to bf16 (round to nearest even), as the GEMM outputs are.

Parity: pinned in tests/test_oracle_act.py (the odd-part identity SiLU(v) - SiLU(-v) = v, the
logistic value at 1, both asymptotes, zeros, the gate/up placement, one rounding to bf16).
"""
import numpy as np

from .formats import bf16r


def silu(v):
    """SiLU in fp64; exp overflow for very negative v gives the limit -0."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def silu_mul(gate_up, inter):
    """gate_up [rows][2*inter] (gate | up) -> bf16-rounded SiLU(gate) * up [rows][inter] (float64)."""
    g = np.asarray(gate_up, dtype=np.float64)
    assert g.ndim == 2 and g.shape[1] == 2 * inter
    return bf16r(silu(g[:, :inter]) * g[:, inter:])
