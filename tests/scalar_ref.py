"""Pure-Python scalar restatement of the Q4_K block for brute-force pins.

Written per byte and per bit from the block description (fp16 d at bytes
0-1, fp16 dmin at bytes 2-3, 12 bytes of packed 6-bit scales/mins, 128
bytes of 4-bit quants in four groups of 32), independently of the vectorised
oracle, so that an index or packing slip in either one shows up as a
mismatch on small inputs.
"""
import math
import struct


def half_to_float(lo_byte: int, hi_byte: int) -> float:
    """Decode IEEE binary16 from its two little-endian bytes by hand."""
    bits = lo_byte | (hi_byte << 8)
    sign = -1.0 if bits & 0x8000 else 1.0
    exp = (bits >> 10) & 0x1F
    frac = bits & 0x3FF
    if exp == 0:
        return sign * frac * 2.0 ** -24
    if exp == 31:
        return sign * (math.inf if frac == 0 else math.nan)
    return sign * (1024 + frac) * 2.0 ** (exp - 25)


def scale_min(block: bytes, j: int):
    s = block[4:16]
    if j < 4:
        return s[j] & 0x3F, s[j + 4] & 0x3F
    sc = (s[j + 4] & 0x0F) + 16 * (s[j - 4] >> 6)
    mn = (s[j + 4] >> 4) + 16 * (s[j] >> 6)
    return sc, mn


def weight(block: bytes, i: int) -> float:
    """Value of weight i (0..255) of one 144-byte block, as an exact float."""
    d = half_to_float(block[0], block[1])
    dmin = half_to_float(block[2], block[3])
    group, pos = divmod(i, 64)
    byte = block[16 + 32 * group + (pos % 32)]
    q = (byte & 0x0F) if pos < 32 else (byte >> 4)
    sc, mn = scale_min(block, i // 32)
    return d * sc * q - dmin * mn


def row_weights(row_blocks) -> list:
    out = []
    for blk in row_blocks:
        b = bytes(bytearray(blk))
        out.extend(weight(b, i) for i in range(256))
    return out


def silu(z: float) -> float:
    if z < -700.0:
        return -0.0 if z < 0 else 0.0
    return z / (1.0 + math.exp(-z))


def f32(v: float) -> float:
    return struct.unpack("<f", struct.pack("<f", v))[0]


def q6k_weight(block: bytes, i: int) -> float:
    """Value of weight i (0..255) of one 210-byte Q6_K block, as an exact float.

    Written per byte and bit from the block description (ql[128] low nibbles,
    qh[64] high 2-bit fields, 16 signed scales at byte 192, fp16 d at byte 208).
    """
    d = half_to_float(block[208], block[209])
    h, r = divmod(i, 128)
    s, l = divmod(r, 32)
    byte = block[64 * h + l + 32 * (s % 2)]
    nib = (byte & 0x0F) if s < 2 else (byte >> 4)
    top = (block[128 + 32 * h + l] >> (2 * s)) & 3
    q = nib + 16 * top
    sc = block[192 + i // 16]
    if sc >= 128:
        sc -= 256
    return d * sc * (q - 32)
