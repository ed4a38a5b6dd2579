"""Pins for the oracle's Q8_1 activation quantizer (CPU only)."""
import os

import numpy as np

import oracle
import workloads

from tests.golden_files import q8_1_blocks, q8_1_byte_vector


def test_handmade_blocks():
    blocks = q8_1_blocks()
    assert {"A", "B", "C", "D", "E", "F"} <= set(blocks)
    for name, b in blocks.items():
        q, d, s = oracle.quantize_q8_1(b["x"][None])
        assert np.array_equal(q[0].astype(np.int64), b["q"]), name
        if "d" in b:
            assert d[0, 0] == np.float32(b["d"]) and s[0, 0] == np.float32(b["s"]), name
        if "dbits" in b:
            assert int(d[0, 0:1].view(np.uint32)[0]) == b["dbits"], name
            assert int(s[0, 0:1].view(np.uint32)[0]) == b["sbits"], name


def test_bytes_layout_against_hand_written_vector():
    """The planar byte layout (quants, then {d, s} per block) against bytes written out by hand."""
    x, want = q8_1_byte_vector()
    q, d, s = oracle.quantize_q8_1(x)
    got = oracle.q8_1_to_bytes(q, d, s)
    assert got.dtype == np.uint8 and got.size == want.size
    assert np.array_equal(got, want), f"first mismatch at byte {int(np.argmax(got != want))}"
    q2, d2, s2 = oracle.q8_1_from_bytes(want, 2, 256)
    assert q2[0, 0] == 127 and q2[0, 32] == -127 and q2[0, 33] == 2 and q2[1, 40] == -2 and q2[1, 63] == 127
    assert np.count_nonzero(q2) == 5
    z = [0.0] * 6
    assert d2.tolist() == [[1.0, 0.5] + z, [0.0, 2.0] + z]
    assert s2.tolist() == [[127.0, -62.5] + z, [0.0, 250.0] + z]


def test_single_nonzero_block():
    for v in [3.0e-7, -1.0, 7.25, -900.0, 1.0e9]:
        x = np.zeros((1, 64), np.float32)
        x[0, 37] = v
        q, d, s = oracle.quantize_q8_1(x)
        assert q[0, 37] == (127 if v > 0 else -127)
        assert np.count_nonzero(q) == 1
        assert d[0, 1] == np.float32(abs(np.float32(v))) / np.float32(127)
        assert d[0, 0] == 0 and s[0, 0] == 0
        assert s[0, 1] == np.float32(d[0, 1] * np.float32(q[0, 37]))


def test_error_bound_and_range():
    xf, _ = workloads.activations(workloads.CONFIGS[3], m=16)
    q, d, s = oracle.quantize_q8_1(xf)
    assert np.abs(q.astype(np.int64)).max() <= 127
    deq = oracle.dequantize_q8_1(q, d)
    step = np.repeat(d.astype(np.float64), 32, axis=1)
    # half a step, plus the two float32 roundings in inv = 127/amax and x*inv
    # (each at most 2^-24 relative on a value of magnitude <= 127 steps)
    assert np.all(np.abs(deq - xf) <= 0.5 * step + 127.0 * step * 2.0 ** -22)
    # the block maximum is always reached with |q| == 127
    amax_pos = np.abs(xf.reshape(16, -1, 32)).argmax(axis=-1)
    qq = np.abs(q.reshape(16, -1, 32).astype(np.int64))
    assert np.all(np.take_along_axis(qq, amax_pos[..., None], -1) == 127)


def test_sum_field_is_scaled_integer_sum():
    xf, _ = workloads.activations(workloads.CONFIGS[2], m=2)
    q, d, s = oracle.quantize_q8_1(xf)
    isum = q.reshape(2, -1, 32).astype(np.int64).sum(-1)
    assert np.all(np.abs(isum) <= 32 * 127)
    # s/d recovers the integer sum up to one float32 rounding of s
    nz = d > 0
    ratio = s[nz].astype(np.float64) / d[nz].astype(np.float64)
    assert np.all(np.abs(ratio - isum[nz]) <= np.abs(isum[nz]) * 2.0 ** -23 + 1e-12)


def test_bytes_roundtrip():
    xf, _ = workloads.activations(workloads.CONFIGS[0], m=3)
    q, d, s = oracle.quantize_q8_1(xf)
    buf = oracle.q8_1_to_bytes(q, d, s)
    assert buf.size == 3 * 256 + 3 * 8 * 8
    q2, d2, s2 = oracle.q8_1_from_bytes(buf, 3, 256)
    assert np.array_equal(q, q2) and np.array_equal(d, d2) and np.array_equal(s, s2)
