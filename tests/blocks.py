"""Hand-built GGUF blocks for the oracle pins.

Each builder writes the bytes of one block from chosen field values, following
the layout statements of the kernel sources on "ferrox-cuda 0.14.0 —
src/gpu.rs" (block structure, nibble/bit-plane positions, the 6-bit
scale/min packing).  The packing of scales is the inverse of the page's
ferrox_q4_k_scale_min (the page gives only the unpacking); the tests pin
pack-then-unpack exhaustively.
"""
import numpy as np


def f16_bits(v: float) -> int:
    return int(np.array([v], dtype="<f2").view("<u2")[0])


def put16(b: bytearray, off: int, bits: int):
    b[off] = bits & 0xFF
    b[off + 1] = (bits >> 8) & 0xFF


def pack_k_scales(sc, m) -> bytes:
    """12 bytes holding eight 6-bit (scale, min) pairs."""
    s = bytearray(12)
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
    for j in range(4, 8):
        s[j + 4] = (sc[j] & 15) | ((m[j] & 15) << 4)
    return bytes(s)


def q8_0(d_bits: int, q) -> bytes:
    b = bytearray(34)
    put16(b, 0, d_bits)
    for i in range(32):
        b[2 + i] = int(q[i]) & 0xFF
    return bytes(b)


def q4_0(d_bits: int, nib) -> bytes:
    """nib[32] in 0..15: element i < 16 is the low nibble of byte i,
    element i >= 16 the high nibble of byte i-16."""
    b = bytearray(18)
    put16(b, 0, d_bits)
    for i in range(16):
        b[2 + i] = (nib[i] & 15) | ((nib[i + 16] & 15) << 4)
    return bytes(b)


def q4_k(d_bits: int, dmin_bits: int, sc, m, q) -> bytes:
    """q[256] in 0..15; group oi: byte 32oi+l low nibble = element 64oi+l,
    high nibble = element 64oi+32+l."""
    b = bytearray(144)
    put16(b, 0, d_bits)
    put16(b, 2, dmin_bits)
    b[4:16] = pack_k_scales(sc, m)
    for oi in range(4):
        for l in range(32):
            b[16 + 32 * oi + l] = (q[64 * oi + l] & 15) | ((q[64 * oi + 32 + l] & 15) << 4)
    return bytes(b)


def q5_k(d_bits: int, dmin_bits: int, sc, m, q) -> bytes:
    """q[256] in 0..31: low 4 bits as Q4_K (qs @48), bit 4 in qh[l] bit 2oi
    (element 64oi+l) or bit 2oi+1 (element 64oi+32+l)."""
    b = bytearray(176)
    put16(b, 0, d_bits)
    put16(b, 2, dmin_bits)
    b[4:16] = pack_k_scales(sc, m)
    for oi in range(4):
        for l in range(32):
            lo, hi = q[64 * oi + l], q[64 * oi + 32 + l]
            b[48 + 32 * oi + l] = (lo & 15) | ((hi & 15) << 4)
            b[16 + l] |= ((lo >> 4) & 1) << (2 * oi)
            b[16 + l] |= ((hi >> 4) & 1) << (2 * oi + 1)
    return bytes(b)


def q6_k(d_bits: int, scales, v) -> bytes:
    """v[256] in 0..63 (the stored 6-bit value; the weight uses v-32);
    scales[16] int8.  Half h, l < 32: ql[64h+l] holds elements 128h+l (low
    nibble) and 128h+l+64 (high); ql[64h+32+l] holds 128h+l+32 and
    128h+l+96; qh[32h+l] bit pairs 0-1, 2-3, 4-5, 6-7 hold the top two bits of
    elements +0, +32, +64, +96."""
    b = bytearray(210)
    for h in range(2):
        for l in range(32):
            e0, e1, e2, e3 = (128 * h + l + 32 * t for t in range(4))
            b[64 * h + l] = (v[e0] & 15) | ((v[e2] & 15) << 4)
            b[64 * h + 32 + l] = (v[e1] & 15) | ((v[e3] & 15) << 4)
            b[128 + 32 * h + l] = ((v[e0] >> 4) & 3) | (((v[e1] >> 4) & 3) << 2) | \
                (((v[e2] >> 4) & 3) << 4) | (((v[e3] >> 4) & 3) << 6)
    for i in range(16):
        b[192 + i] = int(scales[i]) & 0xFF
    put16(b, 208, d_bits)
    return bytes(b)
