"""Pins for the oracle's Q6_K block decoding and GEMV (CPU only)."""
import os

import numpy as np

import oracle
import workloads
from tests import scalar_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _handmade():
    blk = np.zeros(210, dtype=np.uint8)
    expect = {}
    for line in open(os.path.join(GOLDEN, "q6k_handmade_block.txt")):
        f = line.split("#")[0].split()
        if not f:
            continue
        if f[0] == "d_bits":
            v = int(f[1], 16)
            blk[208], blk[209] = v & 0xFF, v >> 8
        elif f[0] == "scale_bytes":
            blk[192:208] = [int(b, 16) for b in f[1:]]
        elif f[0] == "set":
            base = 0 if f[1] == "ql" else 128
            blk[base + int(f[2])] = int(f[3], 16)
        elif f[0] == "expect":
            expect[int(f[1])] = float(f[2])
    return blk, expect


def test_handmade_block_values():
    blk, expect = _handmade()
    w = oracle.dequantize_q6k(blk[None, None])[0]
    sc = blk[192:208].view(np.int8).astype(np.float64)
    for i in range(256):
        want = expect.get(i, sc[i // 16] * -32.0)   # unlisted weights have q = 0
        assert w[i] == want, (i, w[i], want)


def test_scalar_decoder_agrees_on_random_blocks():
    """Per-weight scalar decoding against the vectorised oracle, every weight of 24 random blocks."""
    blocks = workloads.q6k_blocks(7, 1, 4, 6 * 256)
    w = oracle.dequantize_q6k(blocks)
    for r in range(4):
        for b in range(6):
            blk = bytes(blocks[r, b].tobytes())
            ref = [scalar_ref.q6k_weight(blk, i) for i in range(256)]
            assert np.array_equal(w[r, 256 * b:256 * (b + 1)], np.array(ref))


def test_weights_exact_in_float32():
    w = oracle.dequantize_q6k(workloads.q6k_blocks(3, 1, 16, 1024))
    assert np.array_equal(w.astype(np.float32).astype(np.float64), w)


def test_gemv_brute_force_tiny():
    blocks = workloads.q6k_blocks(11, 1, 6, 512)
    x = workloads.normal(11, 4, 3 * 512).reshape(3, 512).astype(np.float32)
    y = oracle.gemv_q6k(x, blocks)
    for t in range(3):
        for n in range(6):
            ws = []
            for b in range(2):
                blk = bytes(blocks[n, b].tobytes())
                ws.extend(scalar_ref.q6k_weight(blk, i) for i in range(256))
            acc = 0.0
            for k in range(512):
                acc += ws[k] * float(x[t, k])
            assert abs(y[t, n] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_quant_32_and_zero_scales_give_zero():
    blocks = workloads.q6k_blocks(5, 1, 8, 512)
    mid = blocks.copy()
    mid[..., 0:128] = 0x00
    mid[..., 128:192] = 0xAA          # every 2-bit field 2: q = 32
    x = workloads.normal(5, 4, 512).reshape(1, 512).astype(np.float32)
    assert np.count_nonzero(oracle.gemv_q6k(x, mid)) == 0
    zs = blocks.copy()
    zs[..., 192:208] = 0
    assert np.count_nonzero(oracle.gemv_q6k(x, zs)) == 0


def test_linear_in_d_and_scales():
    blocks = workloads.q6k_blocks(9, 1, 8, 768)
    x = workloads.normal(9, 4, 2 * 768).reshape(2, 768).astype(np.float32)
    y = oracle.gemv_q6k(x, blocks)
    dbl = blocks.copy()
    d = dbl[..., 208:210].copy().view(np.float16) * np.float16(2.0)  # exact: one exponent step
    dbl[..., 208:210] = d.view(np.uint8)
    assert np.allclose(oracle.gemv_q6k(x, dbl), 2.0 * y, rtol=1e-13, atol=0)
    neg = blocks.copy()
    sc = neg[..., 192:208].view(np.int8).copy()
    sc[sc == -128] = -127
    base = neg.copy()
    base[..., 192:208] = sc.view(np.uint8)
    neg[..., 192:208] = (-sc).view(np.uint8)
    assert np.allclose(oracle.gemv_q6k(x, neg), -oracle.gemv_q6k(x, base), rtol=1e-13, atol=0)


def test_one_hot_rows_gather_x():
    """d = 1, scales 1, q = 32 everywhere except q = 33 at one input per row: y = x[:, src]."""
    n, k = 40, 768
    rng = np.random.default_rng(2)
    blocks = np.zeros((n, k // 256, 210), dtype=np.uint8)
    blocks[..., 128:192] = 0xAA                       # q = 32 everywhere
    blocks[..., 192:208] = 1
    blocks[..., 208:210] = np.frombuffer(np.float16(1.0).tobytes(), dtype=np.uint8)
    src = rng.integers(0, k, size=n)
    for r, c in enumerate(src):
        b, i = divmod(int(c), 256)
        h, rr = divmod(i, 128)
        s, l = divmod(rr, 32)
        byte = 64 * h + l + 32 * (s % 2)
        blocks[r, b, byte] |= 1 if s < 2 else 0x10    # nibble 1 -> q = 33
    x = rng.standard_normal((2, k)).astype(np.float32)
    assert np.array_equal(oracle.gemv_q6k(x, blocks), x[:, src].astype(np.float64))
