"""Pins for the oracle's MoE gather and combine (CPU only): permutation identities against the
routing generator, a hand-computed combine, power-of-two weights (exact in bf16) and empty slots."""
import numpy as np

from moe_hm_gemm_gb300 import synth
from oracle import moe as om


def test_gather_places_each_token_in_its_slots():
    tok, _, _, pos, _ = synth.moe_routing_slots(40, experts=16, topk=4, seed=2)
    x = np.random.default_rng(0).standard_normal((40, 24))
    xs = om.gather_rows(x, tok)
    assert xs.shape == (160, 24)
    for t in range(40):
        for j in range(4):
            np.testing.assert_array_equal(xs[pos[t, j]], x[t])


def test_combine_hand_computed():
    y = np.array([[1.0, 2.0], [4.0, -8.0], [0.5, 0.25]])
    pos = np.array([[1, 0], [2, -1]])
    w = np.array([[0.25, 0.75], [2.0, 9.0]])
    out = om.combine(y, pos, w)
    # token 0: 0.25 * [4, -8] + 0.75 * [1, 2] = [1.75, -0.5]; token 1: 2 * [0.5, 0.25], slot 1 empty
    np.testing.assert_array_equal(out, [[1.75, -0.5], [1.0, 0.5]])


def test_combine_of_gathered_rows_with_unit_weights():
    # identity experts (y = the gathered x) and weights 1: every token is added topk = 8 times,
    # a power of two, so the bf16 result is exactly 8 x
    tok, _, _, pos, _ = synth.moe_routing_slots(30, experts=16, topk=8, seed=3)
    x = np.random.default_rng(1).integers(-64, 64, size=(30, 16)) / 64.0
    out = om.combine(om.gather_rows(x, tok), pos, np.ones((30, 8)))
    np.testing.assert_array_equal(out, 8 * x)


def test_combine_weights_sum_to_one():
    tok, _, _, pos, w = synth.moe_routing_slots(20, experts=8, topk=4, seed=4)
    x = np.random.default_rng(2).integers(-16, 16, size=(20, 8)) / 16.0
    out = om.combine(om.gather_rows(x, tok), pos, w)
    # the float32 weights sum to 1 within a few ulps; one bf16 rounding of x * sum(w)
    assert np.all(np.abs(out - x) <= np.abs(x) * 2.0 ** -8 + 1e-12)
