"""Pins for the oracle's FFN, closed-form block dot product and prefill chain (CPU only)."""
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle
import workloads
from tests import scalar_ref


def _onehot_q4k(rows, cols, pos):
    """Q4_K rows that are unit vectors: d = 1, dmin = 0, every scale 1, q = 1 at pos[r]."""
    nb = cols // 256
    blk = np.zeros((rows, nb, 144), np.uint8)
    blk[:, :, 1] = 0x3C                      # fp16 1.0 = 0x3C00
    blk[:, :, 4:8] = 1                       # scales 0-3 = 1, their top bits 0
    blk[:, :, 12:16] = 1                     # scales 4-7 low nibble = 1, mins 4-7 = 0
    for r in range(rows):
        b, i = divmod(int(pos[r]), 256)
        g, p = divmod(i, 64)
        blk[r, b, 16 + 32 * g + (p % 32)] |= (1 if p < 32 else 16)
    return blk


def test_onehot_weights_make_ffn_a_gather():
    H, I, m = 512, 768, 3
    rng = np.random.default_rng(7)
    pg, pu, pd = rng.integers(0, H, I), rng.integers(0, H, I), rng.integers(0, I, H)
    wg, wu, wd = _onehot_q4k(I, H, pg), _onehot_q4k(I, H, pu), _onehot_q4k(H, I, pd)
    assert np.array_equal(oracle.dequantize_q4k(wg), np.eye(H)[pg])
    x = rng.standard_normal((m, H)).astype(np.float32)
    y, h = oracle.ffn_decode(x, wg, wu, wd)
    g = x[:, pg].astype(np.float64)
    u = x[:, pu].astype(np.float64)
    h_ref = g * expit(g) * u
    assert np.allclose(h, h_ref, rtol=1e-14, atol=0)
    assert np.allclose(y, h_ref[:, pd], rtol=1e-14, atol=0)


def test_onehot_prefill_with_exact_q8_1_inputs():
    """x blocks of integers with |max| = 127 quantize exactly (d = 1), so gate/up gather x."""
    H, I, m = 256, 512, 2
    rng = np.random.default_rng(3)
    pg, pu, pd = rng.integers(0, H, I), rng.integers(0, H, I), rng.integers(0, I, H)
    wg, wu, wd = _onehot_q4k(I, H, pg), _onehot_q4k(I, H, pu), _onehot_q4k(H, I, pd)
    x = rng.integers(-126, 127, (m, H)).astype(np.float32)
    x.reshape(m, -1, 32)[:, :, 0] = 127.0
    out = oracle.ffn_prefill(x, wg, wu, wd)
    xq, xd, _ = out["xq"]
    assert np.array_equal(xq.astype(np.float32), x) and np.all(xd == 1.0)
    g = x[:, pg].astype(np.float64)
    u = x[:, pu].astype(np.float64)
    h = (g * expit(g) * u).astype(np.float32)
    assert np.array_equal(out["h"], h)
    hq, hd, _ = out["hq"]
    assert np.allclose(out["y"], oracle.dequantize_q8_1(hq, hd)[:, pd], rtol=0, atol=0)


def test_zero_input_gives_zero_output():
    c = workloads.small_config(256, 512, 2)
    wg, wu, wd = workloads.weights(c)
    y, h = oracle.ffn_decode(np.zeros((2, 256), np.float32), wg, wu, wd)
    assert np.all(y == 0) and np.all(h == 0)
    out = oracle.ffn_prefill(np.zeros((2, 256), np.float32), wg, wu, wd)
    assert np.all(out["y"] == 0)


def test_decode_matches_scalar_bruteforce():
    H, I, m = 256, 256, 2
    c = workloads.small_config(H, I, m)
    wg, wu, wd = workloads.weights(c)
    x, _ = workloads.activations(c)
    y, h = oracle.ffn_decode(x, wg, wu, wd)
    Wg = [scalar_ref.row_weights(wg[r]) for r in range(I)]
    Wu = [scalar_ref.row_weights(wu[r]) for r in range(I)]
    Wd = [scalar_ref.row_weights(wd[r]) for r in range(H)]
    for t in range(m):
        xs = [float(v) for v in x[t]]
        hh = []
        for i in range(I):
            g = math.fsum(Wg[i][k] * xs[k] for k in range(H))
            u = math.fsum(Wu[i][k] * xs[k] for k in range(H))
            hh.append(scalar_ref.silu(g) * u)
        for n in range(H):
            yy = math.fsum(Wd[n][i] * hh[i] for i in range(I))
            assert abs(yy - y[t, n]) <= 1e-11 * (abs(yy) + 1.0)
        assert np.allclose(h[t], hh, rtol=1e-11)


def test_gate_equal_up_gives_silu_times_gate():
    c = workloads.small_config(256, 512, 1)
    wg, _, wd = workloads.weights(c)
    x, _ = workloads.activations(c)
    _, h = oracle.ffn_decode(x, wg, wg, wd)
    g = x.astype(np.float64) @ oracle.dequantize_q4k(wg).T
    assert np.allclose(h, g * g * expit(g), rtol=1e-12)


def test_closed_form_block_dot():
    """d*sum(scale*d8*sum q4*q8) - dmin*sum(min*s8) equals the dequantized dot product."""
    blocks = workloads.q4k_blocks(11, 1, 6, 256)[:, 0]
    xs, _ = workloads.activations(workloads.small_config(256, 256, 6, "bf16", ("channels", 0.01, 100.0)))
    for b in range(6):
        q8, d8, s8 = oracle.quantize_q8_1(xs[b:b + 1])
        exact_s = d8[0].astype(np.float64) * q8[0].reshape(8, 32).astype(np.int64).sum(1)
        cf = oracle.q4k_q8_1_dot(blocks[b], q8[0], d8[0], exact_s)
        # independent dequantization from the scalar per-byte decoder
        w = np.array(scalar_ref.row_weights([blocks[b]]))
        ref = math.fsum(w * oracle.dequantize_q8_1(q8, d8)[0])
        assert abs(cf - ref) <= 1e-12 * (abs(ref) + 1.0)
        # with the stored float32 sum the min term moves by at most one float32 rounding
        cf32 = oracle.q4k_q8_1_dot(blocks[b], q8[0], d8[0], s8[0])
        d, dmin, sc, mn, _ = oracle.q4k_fields(blocks[b][None])
        bound = sum(float(dmin[0]) * int(mn[0, j]) * abs(float(s8[0, j])) for j in range(8)) * 2.0 ** -23
        assert abs(cf32 - ref) <= bound + 1e-12 * abs(ref)


def test_silu_special_values():
    z = np.array([-1e4, -800.0, 0.0, 1e-300, 5.0, 800.0, 1e4])
    s = oracle.silu(z)
    assert s[0] == 0 and np.signbit(s[0]) and s[1] == 0
    assert s[2] == 0 and s[6] == 1e4 and s[5] == 800.0
    assert np.isclose(s[4], 5.0 * expit(5.0), rtol=1e-15)
