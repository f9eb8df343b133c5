"""Pins for the oracle's number formats (CPU only).

Each test fixes a property from the format's public definition or cross-checks against a
library routine, so that a wrong bias, a wrong field width or a wrong tie rule fails.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F


def test_e2m1_decode_table():
    # OCP MX v1.0 FP4 (E2M1): the eight magnitudes, then the same with the sign bit.
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = F.decode_e2m1(np.arange(16))
    np.testing.assert_array_equal(got[:8], mags)
    np.testing.assert_array_equal(got[8:], [-m for m in mags])
    assert np.signbit(got[8])


def test_e4m3_decode_landmarks():
    d = lambda c: float(F.decode_e4m3(c))
    assert d(0x7E) == 448.0            # largest finite (S.1111.110)
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x38) == 1.0              # exponent field 7 = bias
    assert d(0x08) == 2.0 ** -6        # smallest normal
    assert d(0x01) == 2.0 ** -9        # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9    # largest subnormal
    assert d(0xB8) == -1.0
    finite = F.decode_e4m3(np.arange(127))
    assert np.all(np.diff(finite) > 0)  # codes 0..126 are strictly increasing


def test_e8m0_decode():
    assert float(F.decode_e8m0(127)) == 1.0
    assert float(F.decode_e8m0(0)) == 2.0 ** -127
    assert float(F.decode_e8m0(254)) == 2.0 ** 127
    assert np.isnan(F.decode_e8m0(255))


@pytest.mark.parametrize("dec,enc,codes", [
    (F.decode_e2m1, F.encode_e2m1, np.arange(16)),
    (F.decode_e4m3, F.encode_e4m3, np.r_[np.arange(0x7F), np.arange(0x80, 0xFF)]),
])
def test_round_trip_every_finite_code(dec, enc, codes):
    np.testing.assert_array_equal(enc(dec(codes)), codes)


def test_e2m1_rne_ties_and_saturation():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.25, -5.0, 0.2, 0.3])
    want = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -0.0, -4.0, 0.0, 0.5])
    got = F.round_to(x, F.E2M1, satfinite=True)
    np.testing.assert_array_equal(got, want)
    assert np.signbit(got[9])


def test_e4m3_rounding_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(2000) * 1e-2,
                        np.linspace(-448, 448, 3001)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(F.e4m3_rne(x.astype(np.float64)), ref)


def test_e4m3_satfinite():
    np.testing.assert_array_equal(F.e4m3_rne(np.array([449.0, 464.0, 1e6, -1e6])),
                                  [0x7E, 0x7E, 0x7E, 0xFE])


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(50000), rng.standard_normal(1000) * 1e-38,
                        rng.standard_normal(1000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(F.bf16r(x.astype(np.float64)), ref)


def test_bf16_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7
    assert F.bf16r(one + ulp / 2) == one              # tie, 1.0 has an even last bit
    assert F.bf16r(one + 3 * ulp / 2) == one + 2 * ulp
    assert F.bf16r(one + ulp / 2 + 2.0 ** -30) == one + ulp


def test_f32_matches_numpy_cast():
    x = np.random.default_rng(2).standard_normal(1000) * 1e3
    np.testing.assert_array_equal(F.f32(x), x.astype(np.float32).astype(np.float64))


def test_bf16_bits_round_trip():
    bits = np.random.default_rng(3).integers(0, 0x7F80, size=500).astype(np.uint16)
    np.testing.assert_array_equal(F.bf16_bits(F.decode_bf16_bits(bits)), bits)
