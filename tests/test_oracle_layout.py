"""Pins for the oracle's packed layouts (CPU only): byte accounting from the explainer page,
hand-computed offsets, and pack/unpack round trips on ragged shapes."""
import json
import os

import numpy as np
import pytest

from oracle import layout as L
from oracle import formats as F
from oracle import quant as Q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int4_worked_example.json")


def test_group_accounting_matches_page():
    g = json.load(open(GOLDEN))
    # one unit is 128 rows x (128 INT4 values + one 16-bit scale)
    assert L.unit_bytes(L.FMT_W4A16_INT4, False) == 128 * g["group_bytes"]
    assert g["weight_bytes"] == g["group_values"] * 4 // 8
    assert L.unit_bytes(L.FMT_W4A16_INT4, False) * 8 / (128 * 128) == g["bits_per_value"]
    # with a u4 zero-point per group: 4 + 16/128 + 4/128 bits
    assert L.unit_bytes(L.FMT_W4A16_INT4, True) * 8 / (128 * 128) == 4 + 20 / 128


def test_payload_sizes():
    assert L.payload_bytes(L.FMT_W4A16_MXFP4, 256, 256) == 4 * 8704
    assert L.payload_bytes(L.FMT_W4A8_MXFP4, 4096, 4096) == 4096 * 2048 + 32 * 32 * 512
    assert L.payload_bytes(L.FMT_W4A4_NVFP4, 8192, 8192) == 8192 * 4096 + 64 * 128 * 512
    assert L.packed_size(L.FMT_W4A16_INT4, 130, 128) == 256 + 2 * 8448   # N padded to 256


def test_hand_computed_offsets():
    pos = lambda kk: tuple(int(v) for v in L.nibble_position(kk))
    assert pos(0) == (0, 0)
    assert pos(1) == (2, 0)        # odd k in the high half-word
    assert pos(2) == (0, 4)
    assert pos(3) == (2, 4)
    assert pos(6) == (1, 4)
    assert pos(7) == (3, 4)
    assert pos(8) == (4, 0)
    assert pos(32) == (2048, 0)
    assert pos(127) == (3 * 2048 + 12 + 3, 4)
    assert int(L.atom_offset(0, 0)) == 0
    assert int(L.atom_offset(1, 0)) == 16
    assert int(L.atom_offset(32, 0)) == 4
    assert int(L.atom_offset(33, 2)) == 22
    assert int(L.atom_offset(127, 3)) == 511
    offs = L.atom_offset(np.arange(128)[:, None], np.arange(4)[None, :])
    assert sorted(offs.ravel().tolist()) == list(range(512))   # a permutation of the atom


def test_header_fields():
    buf = L.pack_w4a4_nvfp4(np.zeros((3, 64), np.uint8), np.zeros((3, 4), np.uint8), 0.5)
    h = L.parse_header(buf)
    assert h == dict(magic=L.MAGIC, fmt=4, N=3, K=64, N_pad=128, K_pad=256, has_zero=False,
                     tensor_scale=0.5, payload_bytes=128 * 128 + 4 * 512)
    assert len(buf) == L.packed_size(4, 3, 64)


@pytest.mark.parametrize("has_zero", [False, True])
def test_int4_round_trip(has_zero):
    rng = np.random.default_rng(0)
    n, k = 200, 256
    w = rng.standard_normal((n, k)) * 0.02
    z = rng.integers(0, 16, size=(n, k // 128)) if has_zero else None
    q, s = Q.quant_int4(w, zeros=z)
    buf = L.pack_w4a16_int4(q, s, z)
    assert len(buf) == L.packed_size(1, n, k, has_zero)
    nib, units = L.unpack_units(buf)
    np.testing.assert_array_equal(nib, q if has_zero else q + 8)
    sb = units[:, :, 8192:8448].view(np.uint16)          # [nt, kb, 128]
    got = sb.transpose(0, 2, 1).reshape(-1, k // 128)[:n]
    from oracle.formats import bf16_bits
    np.testing.assert_array_equal(got, bf16_bits(s))
    if has_zero:
        zb = units[:, :, 8448:8512]
        zz = np.stack([zb & 0xF, zb >> 4], axis=-1).reshape(zb.shape[0], zb.shape[1], 128)
        np.testing.assert_array_equal(zz.transpose(0, 2, 1).reshape(-1, k // 128)[:n], z)
    # padded rows are all zero
    assert np.all(units[1, :, :][:, [16 * r for r in range(72, 128)]] == 0)


def test_mxfp4_tiled_round_trip():
    rng = np.random.default_rng(1)
    w = rng.standard_normal((130, 128)) * 0.02
    codes, e = Q.quant_mxfp4(w)
    buf = L.pack_w4a16_mxfp4(codes, e)
    nib, units = L.unpack_units(buf)
    np.testing.assert_array_equal(nib, codes)
    eb = units[:, 0, 8192:8704].reshape(-1, 128, 4).reshape(-1, 4)[:130]
    np.testing.assert_array_equal(eb, e)


def test_mxint4_tiled_round_trip():
    # signed codes are stored biased by 8 (nibble 0 = -8, 8 = 0, 15 = 7); scales as MXFP4
    rng = np.random.default_rng(3)
    w = rng.standard_normal((130, 256)) * 0.02
    q, e = Q.quant_mxint4(w)
    buf = L.pack_w4a16_mxint4(q, e)
    assert len(buf) == L.packed_size(L.FMT_W4A16_MXINT4, 130, 256) == 256 + 2 * 2 * 8704
    nib, units = L.unpack_units(buf)
    np.testing.assert_array_equal(nib, q + 8)
    eb = units[:, :, 8192:8704].reshape(2, 2, 128, 4).transpose(0, 2, 1, 3).reshape(256, 8)[:130]
    np.testing.assert_array_equal(eb, e)
    # one hand-placed code: (row 0, k 33) = -8 -> nibble 0 in the word at byte 2048, bits 16..19
    q2 = np.zeros((1, 128), dtype=np.int64)
    q2[0, 33] = -8
    buf2 = L.pack_w4a16_mxint4(q2, np.zeros((1, 4), dtype=np.int64))
    unit = buf2[256:256 + 8704]
    assert unit[2048 + 2] == 0x80      # low nibble k 33 (q -8 -> 0), high nibble k 35 (q 0 -> 8)
    assert unit[2048 + 3] == 0x88 and unit[2048] == 0x88 and unit[0] == 0x88


@pytest.mark.parametrize("fmt", [3, 4])
def test_rowmajor_round_trip(fmt):
    rng = np.random.default_rng(2)
    n, k = 150, 512
    w = rng.standard_normal((n, k)) * 0.02
    if fmt == 3:
        codes, sf = Q.quant_mxfp4(w)
        buf = L.pack_w4a8_mxfp4(codes, sf)
        chunks = k // 128
    else:
        codes, sf, g = Q.quant_nvfp4(w)
        buf = L.pack_w4a4_nvfp4(codes, sf, g)
        chunks = k // 64
    h = L.parse_header(buf)
    body_len = h["N_pad"] * h["K_pad"] // 2
    body = buf[L.HEADER:L.HEADER + body_len]
    np.testing.assert_array_equal(L.unpack_codes_rowmajor(body, h["N_pad"], k)[:n], codes)
    atoms = buf[L.HEADER + body_len:]
    np.testing.assert_array_equal(L.unpack_atoms(atoms, n, chunks), np.asarray(sf, np.uint8))


def test_act_nvfp4_layout():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((70, 128))
    codes, sb, g = Q.quant_nvfp4(x)
    body, atoms = L.pack_act_nvfp4(codes, sb)
    assert body.shape == (70, 64) and atoms.size == L.act_scale_bytes(70, 128) == 2 * 512
    np.testing.assert_array_equal(L.unpack_codes_rowmajor(body, 70, 128), codes)
    np.testing.assert_array_equal(L.unpack_atoms(atoms, 70, 2), sb)


@pytest.mark.parametrize("group,has_zero", [(32, True), (64, True), (32, False)])
def test_int4_g32_units(group, has_zero):
    """Per-32 INT4 units: nibbles as INT4, the bf16 scale of (r, chunk c) at 8192 + 8r + 2c and its
    zero-point nibble at 9216 + 2r + c // 2, bit 4 (c % 2); a group of 64 fills two chunks."""
    from oracle.formats import bf16_bits
    rng = np.random.default_rng(9)
    w = rng.standard_normal((130, 256)) * 0.02
    z = rng.integers(0, 16, size=(130, 256 // group)) if has_zero else None
    q, s = Q.quant_int4(w, zeros=z, group=group)
    buf = L.pack_w4a16_int4_g32(q, s, z, group=group)
    assert len(buf) == L.packed_size(L.FMT_W4A16_INT4_G32, 130, 256, has_zero) == 256 + 2 * 2 * (9472 if has_zero else 9216)
    nib, units = L.unpack_units(buf)
    np.testing.assert_array_equal(nib, q if has_zero else q + 8)
    ub = 9472 if has_zero else 9216
    units = units.reshape(2, 2, ub)
    row, kk = 129, 200                       # n-tile 1, k-block 1, chunk (200 % 128) // 32 = 2
    unit = units[1, 1]
    rr, c = row - 128, (kk % 128) // 32
    sb = int(unit[8192 + 8 * rr + 2 * c]) | (int(unit[8192 + 8 * rr + 2 * c + 1]) << 8)
    assert sb == int(bf16_bits(s[row, kk // group]))
    if has_zero:
        zn = (int(unit[9216 + 2 * rr + c // 2]) >> (4 * (c % 2))) & 0xF
        assert zn == z[row, kk // group]


@pytest.mark.parametrize("group", [256, 512])
def test_int4_wide_group_units_carry_their_group_scale(group):
    """A group of 128 j along K fills j consecutive units: unit (t, b) holds the bf16 scale and
    zero-point of group (b * 128) // group for every row, at the INT4 unit offsets."""
    rng = np.random.default_rng(3)
    n, k = 130, 1024
    w = rng.standard_normal((n, k)).astype(np.float32)
    z = rng.integers(0, 16, size=(n, k // group))
    q, s = Q.quant_int4(w, zeros=z, group=group)
    buf = L.pack_w4a16_int4(q, s, z, group=group)
    assert len(buf) == L.packed_size(1, n, k, True)
    kb = k // 128
    for row, b in [(0, 0), (129, kb - 1), (77, 3), (5, 1)]:
        unit = 256 + ((row // 128) * kb + b) * 8512
        r = row % 128
        sb = int(buf[unit + 8192 + 2 * r]) | (int(buf[unit + 8192 + 2 * r + 1]) << 8)
        assert sb == int(F.bf16_bits(s[row, (b * 128) // group]))
        zn = (int(buf[unit + 8448 + r // 2]) >> (4 * (r % 2))) & 0xF
        assert zn == z[row, (b * 128) // group]


@pytest.mark.parametrize("has_zero", [False, True])
def test_int8_units(has_zero):
    """Format 7 units: code bytes at (kk // 16) * 2048 + r * 16 + kk % 16 (q + 128 without zero-points),
    the row's bf16 scale at 16384 + 2r, its zero-point at 16640 + r; a round trip through the offsets."""
    rng = np.random.default_rng(5)
    n, k = 130, 256
    w = rng.standard_normal((n, k)).astype(np.float32)
    z = rng.integers(0, 256, size=(n, k // 128)) if has_zero else None
    q, s = Q.quant_int8(w, zeros=z)
    buf = L.pack_w8a16_int8(q, s, z)
    assert len(buf) == L.packed_size(7, n, k, has_zero) == 256 + 2 * 2 * (16768 if has_zero else 16640)
    ub = L.unit_bytes(7, has_zero)
    for row, kk in [(0, 0), (5, 17), (129, 255), (77, 130), (127, 127)]:
        unit = 256 + ((row // 128) * (k // 128) + kk // 128) * ub
        r, c = row % 128, kk % 128
        code = int(buf[unit + (c // 16) * 2048 + r * 16 + c % 16])
        assert code == (q[row, kk] if has_zero else q[row, kk] + 128)
        sb = int(buf[unit + 16384 + 2 * r]) | (int(buf[unit + 16384 + 2 * r + 1]) << 8)
        assert sb == int(F.bf16_bits(s[row, kk // 128]))
        if has_zero:
            assert int(buf[unit + 16640 + r]) == z[row, kk // 128]
