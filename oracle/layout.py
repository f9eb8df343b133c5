"""Byte layout of the preprocessed ("packed") weight and of the quantized activations.

Test infrastructure: an independent statement of the layout that ``hm_transform`` and the
activation quantizers must produce byte for byte. The explainer page ("vLLM Humming은
4비트를 어떻게 계산하나", section "표현을 맞춘 다음 GPU가 읽기 좋은 배치로 바꾼다") says only
that weights, scales and zero-points are first put in a common representation and then
padded and rearranged once into a device-friendly order; the concrete order below is this
library's own design and is documented in include/hm.h.

Packed weight = 256-byte header + payload.

Header (little endian): u32 magic 0x31574D48, u32 fmt, i64 N, i64 K, i64 N_pad, i64 K_pad,
u32 has_zero, f32 tensor_scale, u64 payload_bytes, zeros up to 256 bytes.

Formats: 1 = W4A16 INT4 (group 128, bf16 scales, optional u4 zero-points),
2 = W4A16 MXFP4 (e2m1 + E8M0/32, bf16 activations), 3 = W4A8 MXFP4, 4 = W4A4 NVFP4,
5 = W4A16 MXINT4 (signed int4 + E8M0/32, bf16 activations), 6 = W4A16 INT4 with bf16 scales (and
optional u4 zero-points) per 32 along K (inputs grouped by 32 or 64), 7 = W8A16 INT8 (8-bit codes,
bf16 scale per 128, optional u8 zero-point).

Tiled payload (formats 1, 2, 5, 6): one "unit" per (n_tile of 128 rows, k_block of 128),
n_tile-major. Inside a unit, row r in 0..127 and kk in 0..127:
  * nibble of (r, kk) lives in the 32-bit little-endian word at byte
    (kk//32)*2048 + r*16 + ((kk%32)//8)*4, at bit 4*((kk%8)//2) + 16*(kk%2);
  * format 1: stored nibble u = q + 8 (symmetric) or q (with zero-points); bf16 scale of
    row r at byte 8192 + 2r; zero-point of row r (if any) at byte 8448 + r//2, bit 4*(r%2);
    unit = 8448 bytes, or 8512 with zero-points;
  * format 2: nibble = e2m1 code; E8M0 code of (r, kk//32) at byte 8192 + 4r + kk//32;
    unit = 8704 bytes;
  * format 5: nibble u = q + 8; E8M0 codes as format 2; unit = 8704 bytes;
  * format 6: nibbles as format 1; bf16 scale of (r, kk//32) at byte 8192 + 8r + 2(kk//32); zero-point
    of (r, kk//32) (if any) at byte 9216 + 2r + (kk//32)//2, bit 4((kk//32)%2); unit = 9216 bytes, or
    9472 with zero-points.
  * format 7: one byte per code at (kk//16)*2048 + r*16 + kk%16 (stored q + 128 without zero-points);
    bf16 scale of row r at 16384 + 2r; u8 zero-point at 16640 + r; unit = 16640 bytes, or 16768.

Row-major payload (formats 3, 4): codes as bytes [N_pad][K_pad/2] (even k in the low
nibble), then scale-factor atoms of 512 bytes, atom (n_tile, kc) n_tile-major, where kc
counts chunks of 128 K (format 3, E8M0 per 32) or 64 K (format 4, e4m3 per 16); inside an
atom the scale of (row r, sub-block j in 0..3) is at byte (r%32)*16 + (r//32)*4 + j.

Padding: N_pad = ceil(N/128)*128; K_pad = K (formats 1-3 and 5, K % 128 == 0) or
ceil(K/256)*256 (format 4, K % 64 == 0); padded codes, scales and zero-points are zero.

Quantized activations: FP8 per token is e4m3 bytes [M][K] plus fp32 s_tok [M]; NVFP4 is
codes [M][K/2] (even k low nibble) plus e4m3 scale atoms [ceil(M/128)][K/64] x 512 bytes
with the same in-atom order as above (row = token).

Parity: pinned in tests/test_oracle_layout.py by unpack(pack(.)) round trips, the byte
accounting of the explainer page (128 INT4 values + one 16-bit scale = 66 bytes) and
hand-computed offsets.
"""
import struct

import numpy as np

from .formats import bf16_bits

MAGIC = 0x31574D48
HEADER = 256
FMT_W4A16_INT4, FMT_W4A16_MXFP4, FMT_W4A8_MXFP4, FMT_W4A4_NVFP4, FMT_W4A16_MXINT4 = 1, 2, 3, 4, 5
FMT_W4A16_INT4_G32 = 6
FMT_W8A16_INT8 = 7
TILED = (FMT_W4A16_INT4, FMT_W4A16_MXFP4, FMT_W4A16_MXINT4, FMT_W4A16_INT4_G32, FMT_W8A16_INT8)
TILE_N = 128
ATOM = 512


def padded_dims(fmt, n, k):
    n_pad = -(-n // TILE_N) * TILE_N
    if fmt == FMT_W4A4_NVFP4:
        k_pad = -(-k // 256) * 256
    else:
        k_pad = k
    return n_pad, k_pad


def unit_bytes(fmt, has_zero):
    if fmt == FMT_W4A16_INT4:
        return 8512 if has_zero else 8448
    if fmt in (FMT_W4A16_MXFP4, FMT_W4A16_MXINT4):
        return 8704
    if fmt == FMT_W4A16_INT4_G32:
        return 9472 if has_zero else 9216
    if fmt == FMT_W8A16_INT8:
        return 16768 if has_zero else 16640
    raise ValueError(fmt)


def payload_bytes(fmt, n, k, has_zero=False):
    n_pad, k_pad = padded_dims(fmt, n, k)
    if fmt in TILED:
        return (n_pad // 128) * (k_pad // 128) * unit_bytes(fmt, has_zero)
    chunk = 128 if fmt == FMT_W4A8_MXFP4 else 64
    return n_pad * k_pad // 2 + (n_pad // 128) * (k_pad // chunk) * ATOM


def packed_size(fmt, n, k, has_zero=False):
    return HEADER + payload_bytes(fmt, n, k, has_zero)


def header(fmt, n, k, has_zero, tensor_scale):
    n_pad, k_pad = padded_dims(fmt, n, k)
    h = struct.pack("<IIqqqqIfQ", MAGIC, fmt, n, k, n_pad, k_pad, int(bool(has_zero)),
                    float(tensor_scale), payload_bytes(fmt, n, k, has_zero))
    return np.frombuffer(h + bytes(HEADER - len(h)), dtype=np.uint8).copy()


# ------------------------------------------------------------------ tiled units (formats 1, 2, 5)

def nibble_position(kk):
    """(byte offset within the nibble region for row 0, bit shift) of column kk in a unit."""
    kk = np.asarray(kk)
    word = (kk // 32) * 2048 + ((kk % 32) // 8) * 4
    bit = 4 * ((kk % 8) // 2) + 16 * (kk % 2)
    return word + bit // 8, bit % 8


def _pack_units(fmt, nibbles, scale_bytes_fn, zeros, n, k, has_zero):
    """nibbles: [N_pad, K_pad] ints 0..15; returns payload bytes."""
    n_pad, k_pad = padded_dims(fmt, n, k)
    ub = unit_bytes(fmt, has_zero)
    nt, kb = n_pad // 128, k_pad // 128
    out = np.zeros((nt, kb, ub), dtype=np.uint8)
    r = np.arange(128)[:, None]
    kk = np.arange(128)[None, :]
    byte, shift = nibble_position(kk)
    off = r * 16 + byte                                  # [128,128] byte offsets
    for t in range(nt):
        for b in range(kb):
            tile = nibbles[t * 128:(t + 1) * 128, b * 128:(b + 1) * 128].astype(np.uint16)
            unit = np.zeros(ub, dtype=np.uint16)
            np.add.at(unit, off.ravel(), (tile << shift).ravel())
            scale_bytes_fn(unit, t, b)
            if has_zero and fmt == FMT_W4A16_INT4:
                zr = zeros[t * 128:(t + 1) * 128, b].astype(np.uint16)
                np.add.at(unit, 8448 + np.arange(128) // 2, zr << (4 * (np.arange(128) % 2)))
            out[t, b] = unit.astype(np.uint8)
    return out.reshape(-1)


def pack_w4a16_int4(q, s, zeros=None, group=128):
    """q int [N,K] (signed without zero-points, unsigned with), s bf16 values [N,K/group],
    zeros ints [N,K/group] or None, group a multiple of 128 dividing K (a group of 128 j gives each
    of its j units its scale and zero-point). Returns the packed buffer (uint8)."""
    q = np.asarray(q)
    n, k = q.shape
    rep = group // 128
    s = np.repeat(np.asarray(s), rep, axis=1)
    if zeros is not None:
        zeros = np.repeat(np.asarray(zeros), rep, axis=1)
    has_zero = zeros is not None
    n_pad, k_pad = padded_dims(FMT_W4A16_INT4, n, k)
    nib = np.zeros((n_pad, k_pad), dtype=np.int64)
    nib[:n, :k] = q if has_zero else q + 8
    sbits = np.zeros((n_pad, k_pad // 128), dtype=np.uint16)
    sbits[:n] = bf16_bits(s)
    z = np.zeros((n_pad, k_pad // 128), dtype=np.int64)
    if has_zero:
        z[:n] = zeros

    def scales(unit, t, b):
        v = sbits[t * 128:(t + 1) * 128, b]
        unit[8192 + 2 * np.arange(128)] = v & 0xFF
        unit[8192 + 2 * np.arange(128) + 1] = v >> 8

    pay = _pack_units(FMT_W4A16_INT4, nib, scales, z, n, k, has_zero)
    return np.concatenate([header(FMT_W4A16_INT4, n, k, has_zero, 1.0), pay])


def pack_w4a16_int4_g32(q, s, zeros=None, group=32):
    """q int [N,K] (signed without zero-points, unsigned with), s bf16 values [N,K/group], zeros ints
    [N,K/group] or None, group 32 or 64 (a group of 64 fills two 32-K chunks). Returns the packed
    buffer (uint8)."""
    q = np.asarray(q)
    n, k = q.shape
    has_zero = zeros is not None
    rep = group // 32
    n_pad, k_pad = padded_dims(FMT_W4A16_INT4_G32, n, k)
    nib = np.zeros((n_pad, k_pad), dtype=np.int64)
    nib[:n, :k] = q if has_zero else q + 8
    sbits = np.zeros((n_pad, k_pad // 32), dtype=np.uint16)
    sbits[:n] = np.repeat(bf16_bits(s), rep, axis=1)
    z = np.zeros((n_pad, k_pad // 32), dtype=np.int64)
    if has_zero:
        z[:n] = np.repeat(np.asarray(zeros, dtype=np.int64), rep, axis=1)
    ub = unit_bytes(FMT_W4A16_INT4_G32, has_zero)
    r = np.arange(128)

    def scales(unit, t, b):
        blk = sbits[t * 128:(t + 1) * 128, b * 4:(b + 1) * 4]        # [128, 4]
        off = 8192 + 8 * r[:, None] + 2 * np.arange(4)[None, :]
        unit[off] = blk & 0xFF
        unit[off + 1] = blk >> 8
        if has_zero:
            zb = z[t * 128:(t + 1) * 128, b * 4:(b + 1) * 4]          # [128, 4]
            unit[9216 + 2 * r] = zb[:, 0] | (zb[:, 1] << 4)
            unit[9216 + 2 * r + 1] = zb[:, 2] | (zb[:, 3] << 4)

    pay = _pack_units(FMT_W4A16_INT4_G32, nib, scales, None, n, k, has_zero)
    assert pay.size == (n_pad // 128) * (k_pad // 128) * ub
    return np.concatenate([header(FMT_W4A16_INT4_G32, n, k, has_zero, 1.0), pay])


def int8_position(kk):
    """Byte offset, within a unit's code region for row 0, of column kk of an INT8 unit: 16-column
    chunks, each chunk 16 contiguous bytes per row, rows 16 bytes apart."""
    kk = np.asarray(kk)
    return (kk // 16) * 2048 + kk % 16


def pack_w8a16_int8(q, s, zeros=None):
    """q int [N,K] (signed in [-128, 127] without zero-points, unsigned in [0, 255] with), s bf16
    values [N,K/128], zeros ints [N,K/128] or None. Units of 128 rows x 128 K: code (r, kk) as a byte
    at (kk//16)*2048 + r*16 + kk%16 (stored q + 128 without zero-points), the bf16 scale of row r at
    16384 + 2r, its u8 zero-point (if any) at 16640 + r. Returns the packed buffer (uint8)."""
    q = np.asarray(q)
    n, k = q.shape
    has_zero = zeros is not None
    n_pad, k_pad = padded_dims(FMT_W8A16_INT8, n, k)
    codes = np.zeros((n_pad, k_pad), dtype=np.int64)
    codes[:n, :k] = q if has_zero else q + 128
    sbits = np.zeros((n_pad, k_pad // 128), dtype=np.uint16)
    sbits[:n] = bf16_bits(s)
    z = np.zeros((n_pad, k_pad // 128), dtype=np.int64)
    if has_zero:
        z[:n] = zeros
    ub = unit_bytes(FMT_W8A16_INT8, has_zero)
    nt, kb = n_pad // 128, k_pad // 128
    out = np.zeros((nt, kb, ub), dtype=np.uint8)
    r = np.arange(128)
    off = r[:, None] * 16 + int8_position(np.arange(128))[None, :]
    for t in range(nt):
        for b in range(kb):
            unit = out[t, b]
            unit[off.ravel()] = codes[t * 128:(t + 1) * 128, b * 128:(b + 1) * 128].ravel().astype(np.uint8)
            v = sbits[t * 128:(t + 1) * 128, b]
            unit[16384 + 2 * r] = v & 0xFF
            unit[16384 + 2 * r + 1] = v >> 8
            if has_zero:
                unit[16640 + r] = z[t * 128:(t + 1) * 128, b]
    return np.concatenate([header(FMT_W8A16_INT8, n, k, has_zero, 1.0), out.reshape(-1)])


def _pack_e8_units(fmt, nibbles, e):
    """Units of 4-bit nibbles [N,K] (0..15) with E8M0 codes [N,K/32] (formats 2 and 5)."""
    nibbles = np.asarray(nibbles)
    n, k = nibbles.shape
    n_pad, k_pad = padded_dims(fmt, n, k)
    nib = np.zeros((n_pad, k_pad), dtype=np.int64)
    nib[:n, :k] = nibbles
    ecodes = np.zeros((n_pad, k_pad // 32), dtype=np.int64)
    ecodes[:n] = e

    def scales(unit, t, b):
        blk = ecodes[t * 128:(t + 1) * 128, b * 4:(b + 1) * 4]      # [128, 4]
        unit[8192 + 4 * np.arange(128)[:, None] + np.arange(4)[None, :]] = blk

    pay = _pack_units(fmt, nib, scales, None, n, k, False)
    return np.concatenate([header(fmt, n, k, False, 1.0), pay])


def pack_w4a16_mxfp4(codes, e):
    """e2m1 codes [N,K] and E8M0 codes [N,K/32] -> packed buffer (uint8)."""
    return _pack_e8_units(FMT_W4A16_MXFP4, codes, e)


def pack_w4a16_mxint4(q, e):
    """Signed codes q [N,K] in [-8, 7] (stored as q + 8) and E8M0 codes [N,K/32] -> packed buffer."""
    return _pack_e8_units(FMT_W4A16_MXINT4, np.asarray(q, dtype=np.int64) + 8, e)


# ------------------------------------------------------------------ row-major codes + atoms (3, 4)

def pack_codes_rowmajor(codes, rows_pad, k_pad):
    """e2m1 codes [R,K] -> bytes [rows_pad, k_pad/2], even k in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    r, k = codes.shape
    full = np.zeros((rows_pad, k_pad), dtype=np.uint8)
    full[:r, :k] = codes
    return (full[:, 0::2] | (full[:, 1::2] << 4)).astype(np.uint8)


def atom_offset(r, j):
    """Byte offset of (row r in 0..127, sub-block j in 0..3) inside a 512-byte atom."""
    r = np.asarray(r)
    return (r % 32) * 16 + (r // 32) * 4 + np.asarray(j)


def pack_atoms(sf, rows_pad, nchunks):
    """sf: scale codes [R, nchunks*4] -> atoms bytes [rows_pad/128][nchunks][512]."""
    sf = np.asarray(sf, dtype=np.uint8)
    r, c = sf.shape
    full = np.zeros((rows_pad, nchunks * 4), dtype=np.uint8)
    full[:r, :c] = sf
    out = np.zeros((rows_pad // 128, nchunks, ATOM), dtype=np.uint8)
    rr = np.arange(128)[:, None]
    jj = np.arange(4)[None, :]
    off = atom_offset(rr, jj)
    for t in range(rows_pad // 128):
        for ch in range(nchunks):
            out[t, ch][off] = full[t * 128:(t + 1) * 128, ch * 4:(ch + 1) * 4]
    return out.reshape(-1)


def pack_w4a8_mxfp4(codes, e):
    n, k = np.asarray(codes).shape
    n_pad, k_pad = padded_dims(FMT_W4A8_MXFP4, n, k)
    body = pack_codes_rowmajor(codes, n_pad, k_pad).reshape(-1)
    atoms = pack_atoms(e, n_pad, k_pad // 128)
    return np.concatenate([header(FMT_W4A8_MXFP4, n, k, False, 1.0), body, atoms])


def pack_w4a4_nvfp4(codes, sb, g):
    n, k = np.asarray(codes).shape
    n_pad, k_pad = padded_dims(FMT_W4A4_NVFP4, n, k)
    body = pack_codes_rowmajor(codes, n_pad, k_pad).reshape(-1)
    atoms = pack_atoms(sb, n_pad, k_pad // 64)
    return np.concatenate([header(FMT_W4A4_NVFP4, n, k, False, g), body, atoms])


# ------------------------------------------------------------------ unpacking (for round trips)

def parse_header(buf):
    magic, fmt, n, k, n_pad, k_pad, hz, ts, pb = struct.unpack("<IIqqqqIfQ", bytes(buf[:struct.calcsize("<IIqqqqIfQ")]))
    return dict(magic=magic, fmt=fmt, N=n, K=k, N_pad=n_pad, K_pad=k_pad, has_zero=bool(hz),
                tensor_scale=ts, payload_bytes=pb)


def unpack_units(buf):
    """Inverse of the tiled layout: returns (nibbles [N,K], scale bytes per unit region)."""
    h = parse_header(buf)
    fmt, n, k = h["fmt"], h["N"], h["K"]
    n_pad, k_pad = h["N_pad"], h["K_pad"]
    ub = unit_bytes(fmt, h["has_zero"])
    units = np.asarray(buf[HEADER:], dtype=np.uint8).reshape(n_pad // 128, k_pad // 128, ub)
    byte, shift = nibble_position(np.arange(128))
    nib = np.zeros((n_pad, k_pad), dtype=np.int64)
    for t in range(n_pad // 128):
        for b in range(k_pad // 128):
            u = units[t, b]
            for r in range(128):
                nib[t * 128 + r, b * 128:(b + 1) * 128] = (u[r * 16 + byte] >> shift) & 0xF
    return nib[:n, :k], units


def unpack_atoms(atoms, rows, nchunks):
    rows_pad = -(-rows // 128) * 128
    a = np.asarray(atoms, dtype=np.uint8).reshape(rows_pad // 128, nchunks, ATOM)
    off = atom_offset(np.arange(128)[:, None], np.arange(4)[None, :])
    out = np.zeros((rows_pad, nchunks * 4), dtype=np.uint8)
    for t in range(rows_pad // 128):
        for ch in range(nchunks):
            out[t * 128:(t + 1) * 128, ch * 4:(ch + 1) * 4] = a[t, ch][off]
    return out[:rows]


def unpack_codes_rowmajor(body, rows, k):
    b = np.asarray(body, dtype=np.uint8).reshape(rows, -1)
    out = np.zeros((rows, b.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out[:, :k]


# ------------------------------------------------------------------ activation layouts

def act_scale_bytes(m, k):
    """Size of the NVFP4 activation scale atoms for an [M,K] activation."""
    return -(-m // 128) * (k // 64) * ATOM


def pack_act_nvfp4(codes, sb):
    m, k = np.asarray(codes).shape
    body = pack_codes_rowmajor(codes, m, k)
    atoms = pack_atoms(sb, -(-m // 128) * 128, k // 64)
    return body, atoms
