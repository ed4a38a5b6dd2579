"""Pins for the oracle's Q4_K block decoding (CPU only)."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from tests import scalar_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_handmade():
    f = {}
    for line in open(os.path.join(GOLDEN, "q4k_handmade_block.txt")):
        line = line.split("#")[0].split()
        if line:
            f[line[0]] = line[1:]
    return f


def _handmade_block():
    f = _read_handmade()
    blk = np.zeros(144, dtype=np.uint8)
    d_bits = int(f["d_bits"][0], 16)
    m_bits = int(f["dmin_bits"][0], 16)
    blk[0], blk[1] = d_bits & 0xFF, d_bits >> 8
    blk[2], blk[3] = m_bits & 0xFF, m_bits >> 8
    blk[4:16] = [int(b, 16) for b in f["scale_bytes"]]
    for i in range(256):
        q = (7 * i + 3) % 16
        g, p = divmod(i, 64)
        idx = 16 + 32 * g + (p % 32)
        if p < 32:
            blk[idx] |= q
        else:
            blk[idx] |= q << 4
    return blk, [int(v) for v in f["scale"]], [int(v) for v in f["min"]]


def test_handmade_block_values():
    blk, sc, mn = _handmade_block()
    w = oracle.dequantize_q4k(blk[None, None])[0]
    expect = [0.5 * sc[i // 32] * ((7 * i + 3) % 16) - 0.25 * mn[i // 32] for i in range(256)]
    assert np.array_equal(w, np.array(expect))


def test_handmade_block_fields():
    blk, sc, mn = _handmade_block()
    d, dmin, s, m, q = oracle.q4k_fields(blk[None])
    assert d[0] == 0.5 and dmin[0] == 0.25
    assert list(s[0]) == sc and list(m[0]) == mn
    assert list(q[0]) == [(7 * i + 3) % 16 for i in range(256)]


def test_scale_packing_is_a_bit_bijection():
    """Each of the 96 packed bits feeds exactly one (field, bit) of the 16 six-bit fields."""
    seen = set()
    for bit in range(96):
        s12 = np.zeros(12, dtype=np.uint8)
        s12[bit // 8] = 1 << (bit % 8)
        sc, mn = oracle.unpack_scales_mins(s12)
        fields = np.concatenate([sc, mn])
        nz = np.nonzero(fields)[0]
        assert len(nz) == 1, bit
        v = int(fields[nz[0]])
        assert v & (v - 1) == 0 and v < 64
        seen.add((int(nz[0]), v.bit_length() - 1))
    assert len(seen) == 96


def test_pack_unpack_all_pairs():
    vals = np.arange(64)
    for j in range(8):
        sc = np.zeros((64, 64, 8), dtype=np.int64)
        mn = np.zeros((64, 64, 8), dtype=np.int64)
        sc[:, :, j] = vals[:, None]
        mn[:, :, j] = vals[None, :]
        # other positions get a fixed pattern so cross-talk would show up
        for jj in range(8):
            if jj != j:
                sc[:, :, jj] = (13 * jj + 5) % 64
                mn[:, :, jj] = (29 * jj + 7) % 64
        s2, m2 = oracle.unpack_scales_mins(oracle.pack_scales_mins(sc, mn))
        assert np.array_equal(s2, sc) and np.array_equal(m2, mn)


def test_dequant_matches_scalar_bruteforce():
    blocks = workloads.q4k_blocks(1234, 1, 3, 768)
    w = oracle.dequantize_q4k(blocks)
    for r in range(3):
        ref = scalar_ref.row_weights(blocks[r])
        assert np.array_equal(w[r], np.array(ref))


def test_dequant_exact_extremes():
    """fp16 subnormal d and the largest dmin still dequantize exactly (rational check)."""
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = [0x01, 0x00]          # d = 2^-24 (smallest subnormal)
    blk[2:4] = [0xFF, 0x7B]          # dmin = 65504
    blk[4:16] = 0xFF                 # all scales and mins = 63
    blk[16:144] = 0xFF               # all quants = 15
    w = oracle.dequantize_q4k(blk[None, None])[0]
    exact = Fraction(1, 2 ** 24) * 63 * 15 - Fraction(65504) * 63
    assert all(Fraction(float(v)) == exact for v in w)
    f32 = oracle.dequantize_q4k_f32(blk[None, None])[0]
    assert np.all(f32 == np.float32(float(exact)))


def test_zero_scales_give_zero():
    blk = np.zeros(144, dtype=np.uint8)
    blk[16:] = 0xAB
    blk[4:16] = 0x3F
    assert np.all(oracle.dequantize_q4k(blk[None, None]) == 0.0)


def test_f32_rounding_is_single_rounding():
    blocks = workloads.q4k_blocks(99, 2, 4, 512)
    exact = oracle.dequantize_q4k(blocks)
    f = oracle.dequantize_q4k_f32(blocks)
    # round-to-nearest: no float32 neighbour is closer to the exact value
    up = np.nextafter(f, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(f, np.float32(-np.inf)).astype(np.float64)
    err = np.abs(f.astype(np.float64) - exact)
    assert np.all(err <= np.abs(up - exact)) and np.all(err <= np.abs(dn - exact))
