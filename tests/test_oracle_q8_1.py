"""Pins for the oracle's Q8_1 activation quantizer (CPU only)."""
import os

import numpy as np

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _blocks():
    out, cur = {}, None
    for line in open(os.path.join(GOLDEN, "q8_1_handmade.txt")):
        t = line.split("#")[0].split()
        if not t:
            continue
        if t[0] == "block":
            cur = {"x": np.zeros(32, np.float32), "q": np.zeros(32, np.int64)}
            out[t[1]] = cur
        elif t[0] == "end":
            cur = None
        elif t[0] in ("d", "s"):
            cur[t[0]] = float(t[1])
        else:
            p = int(t[0])
            cur["x"][p] = np.float32(float(t[1]))
            cur["q"][p] = int(t[2])
    return out


def test_handmade_blocks():
    for name, b in _blocks().items():
        q, d, s = oracle.quantize_q8_1(b["x"][None])
        assert np.array_equal(q[0].astype(np.int64), b["q"]), name
        if "d" in b:
            assert d[0, 0] == np.float32(b["d"]) and s[0, 0] == np.float32(b["s"]), name


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
