"""Pins for the oracle's MoE activation (CPU only): properties of SiLU that fix it without
retyping its formula, the gate/up placement, and one rounding to bf16."""
import numpy as np

from oracle import act as A
from oracle.formats import bf16r


def test_odd_part_identity():
    # SiLU(v) - SiLU(-v) = v for every v: v*sigma(v) - (-v)*sigma(-v) = v*(sigma(v) + sigma(-v))
    v = np.linspace(-20.0, 20.0, 4001)
    np.testing.assert_allclose(A.silu(v) - A.silu(-v), v, rtol=0, atol=1e-12)


def test_logistic_value_at_one_and_zero():
    # sigma(1) = 0.7310585786300049 (the standard logistic at 1), so SiLU(1) equals it
    assert abs(A.silu(1.0) - 0.7310585786300049) < 1e-15
    assert A.silu(0.0) == 0.0


def test_asymptotes():
    # SiLU(v) -> v for large v, -> -0 for very negative v (no overflow error)
    assert abs(A.silu(40.0) - 40.0) < 1e-12
    assert abs(A.silu(-40.0)) < 1e-15
    r = A.silu(np.array([-1e6]))
    assert r[0] == 0.0 and np.signbit(r[0])


def test_gate_first_up_second_and_one_rounding():
    inter = 8
    gate = np.array([[-3.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0, 6.0]])
    up = np.array([[1.0, 2.0, -1.0, 5.0, 3.0, 1.0, -2.0, 0.25]])
    h = A.silu_mul(np.concatenate([gate, up], axis=1), inter)
    # with up = 1 the result is SiLU(gate) rounded to bf16 (a swap would give SiLU(1) * gate)
    ones = A.silu_mul(np.concatenate([gate, np.ones_like(gate)], axis=1), inter)
    np.testing.assert_array_equal(ones, bf16r(A.silu(gate)))
    assert ones[0, 7] != bf16r(A.silu(1.0) * 6.0)
    # every output is a bf16 value, and the product is rounded once (not SiLU rounded first)
    np.testing.assert_array_equal(h, bf16r(h))
    np.testing.assert_array_equal(h, bf16r(A.silu(gate) * up))
