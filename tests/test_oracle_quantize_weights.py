"""Pins for the oracle's min-max Q4_K weight quantizer (CPU only)."""
import numpy as np
import pytest

import oracle
import workloads


def _check_roundtrip(w):
    blocks = oracle.quantize_q4k(w)
    deq = oracle.dequantize_q4k(blocks)
    d, dmin, sc, mn, q = oracle.q4k_fields(blocks)
    step = (d[..., None] * sc).repeat(32, axis=-1).reshape(deq.shape)
    err = np.abs(deq - w.astype(np.float64))
    # half a quant step (plus float64 rounding of the quotient), never more
    assert np.all(err <= 0.5 * step * (1 + 1e-12) + 1e-300)
    assert np.all((q >= 0) & (q <= 15)) and np.all(sc <= 63) and np.all(mn <= 63)
    return blocks


def test_roundtrip_gaussian():
    w = workloads.normal(5, 1, 64 * 512).reshape(64, 512).astype(np.float32)
    _check_roundtrip(w)


def test_roundtrip_mixed_scales_and_signs():
    u = workloads.normal(6, 1, 32 * 1024).reshape(32, 1024)
    scale = np.exp(workloads.normal(6, 2, 32 * 32).reshape(32, 32) * 2.0).repeat(32, axis=1)
    w = (u * scale).astype(np.float32)
    w[0] = np.abs(w[0])          # all positive row
    w[1] = -np.abs(w[1])         # all negative row
    w[2, :256] = 0.0             # an all-zero block
    w[3, 32:64] = 0.0            # an all-zero sub-block
    blocks = _check_roundtrip(w)
    assert np.all(blocks[2, 0, :] == 0)


def test_constant_block():
    w = np.full((1, 256), 1.0, np.float32)
    blocks = _check_roundtrip(w)
    d, dmin, sc, mn, q = oracle.q4k_fields(blocks)
    assert dmin[0, 0] == 0 and np.all(mn == 0)
    # d is the smallest fp16 with 945*d >= 1, and scale 63 gives 15*d*63 >= 1
    assert 945 * d[0, 0] >= 1.0
    prev = np.frombuffer(np.uint16(np.float16(d[0, 0]).view(np.uint16) - 1).tobytes(), np.float16)[0]
    assert 945 * float(prev) < 1.0
    assert np.all(sc == 63) and np.all(q == 15)


def test_overflow_is_an_error():
    with pytest.raises(ValueError):
        oracle.quantize_q4k(np.full((1, 256), 1e8, np.float32))


def test_quantize_dequantize_stable_on_weights():
    """Quantizing dequantized weights again stays within half a step of them."""
    c = workloads.small_config(512, 256, 1)
    wg, _, _ = workloads.weights(c)
    w = oracle.dequantize_q4k_f32(wg)
    _check_roundtrip(w)
