"""MoE token movement around the grouped GEMMs, in fp64 (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU baseline use this module; the product
path never does.

The explainer page ("vLLM Humming은 4비트를 어떻게 계산하나", MoE paragraph of the section "같은
가중치도 한 토큰과 많은 토큰에서 비용이 다르다") has each token routed to some experts, each
expert multiplying its own tokens; the grouped GEMM therefore sees the tokens' rows sorted by
expert. The two steps around it, read as the usual top-k MoE layer (the pages do not print them):

* gather: row r of the expert-sorted activations is token token_of_row[r]'s row;
* combine: token t's output is sum over its routing slots j of w[t, j] times the expert output row
  pos[t, j] (the sorted row of (t, j)), rounded once to bf16; a slot with pos < 0 is empty.

Parity: pinned in tests/test_oracle_moe.py (permutation identities and a hand-built routing).
"""
import numpy as np

from .formats import bf16r


def gather_rows(x, token_of_row):
    """x [T][K] -> [rows][K] with row r = x[token_of_row[r]] (an exact copy)."""
    return np.asarray(x)[np.asarray(token_of_row, dtype=np.int64)]


def combine(y, pos, w):
    """y [rows][N] expert outputs, pos [T][topk] sorted rows (-1 = empty slot), w [T][topk] weights
    -> bf16-rounded [T][N] (float64) of sum_j w[t, j] * y[pos[t, j]]."""
    y = np.asarray(y, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.int64)
    w = np.asarray(w, dtype=np.float64)
    out = np.zeros((pos.shape[0], y.shape[1]))
    for j in range(pos.shape[1]):
        ok = pos[:, j] >= 0
        out[ok] += w[ok, j][:, None] * y[pos[ok, j]]
    return bf16r(out)

