"""Bit-exact GPU tests of Q4_K dequantisation, Q8_1 quantisation and the weight quantizer."""
import numpy as np
import pytest

import oracle
import workloads
from tests.golden_files import q8_1_blocks, q8_1_byte_vector
from tests.gpu_util import dev, lib, to_dev, torch

pytestmark = pytest.mark.gpu


def _adversarial_blocks():
    blk = np.zeros((8, 144), np.uint8)
    rng = np.random.default_rng(1)
    blk[:, 4:] = rng.integers(0, 256, (8, 140), dtype=np.uint8)
    heads = [(0x0000, 0x0000), (0x0001, 0x7BFF), (0x7BFF, 0x0001), (0x03FF, 0x03FF),
             (0x3C00, 0x0000), (0x0000, 0x3C00), (0x8001, 0x0400), (0x1234, 0x5678)]
    for i, (d, m) in enumerate(heads):
        blk[i, 0:2] = [d & 0xFF, d >> 8]
        blk[i, 2:4] = [m & 0xFF, m >> 8]
    blk[1, 4:16] = 0xFF
    blk[1, 16:] = 0xFF
    return blk.reshape(2, 4, 144)


@pytest.mark.parametrize("cfg_index,rows", [(0, None), (1, 512), (2, 512), (3, 256), (4, 256)])
def test_dequant_bit_exact_on_workload_weights(cfg_index, rows):
    cfg = workloads.CONFIGS[cfg_index]
    for mat in workloads.weights(cfg):
        w = mat if rows is None else mat[:rows]
        r, nb, _ = w.shape
        out = lib().q4k_dequantize(to_dev(w), r, nb * 256)
        ref = oracle.dequantize_q4k_f32(w)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_dequant_bit_exact_adversarial():
    w = _adversarial_blocks()
    out = lib().q4k_dequantize(to_dev(w), 2, 1024)
    ref = oracle.dequantize_q4k_f32(w)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def _q8_check(x_f32, x_buf, m, k):
    out = lib().q8_1_quantize_act(to_dev(x_buf))
    q, d, s = oracle.quantize_q8_1(x_f32)
    ref = oracle.q8_1_to_bytes(q, d, s)
    got = out.cpu().numpy()
    assert got.size == ref.size
    assert np.array_equal(got, ref), f"first mismatch at byte {int(np.argmax(got != ref))}"


@pytest.mark.parametrize("cfg_index", [0, 1, 2, 3, 4])
def test_q8_1_bit_exact_on_workload_activations(cfg_index):
    cfg = workloads.CONFIGS[cfg_index]
    m = cfg.m if cfg.m >= 8 else 8
    xf, xb = workloads.activations(cfg, m=m)
    _q8_check(xf, xb, m, cfg.hidden)


def test_q8_1_ties_zero_and_single_blocks():
    x = np.zeros((3, 256), np.float32)
    # block 0 of row 0: amax 127 -> inv 1, exact halves tie away from zero
    x[0, 0:8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -126.5, 3.5]
    # block 1: amax 15.875 -> inv 8, more ties
    x[0, 32:37] = [15.875, 0.0625, -0.1875, 1.3125, -0.3125]
    # row 1: single non-zero entries of various magnitudes
    for j, v in enumerate([3e-7, -1.0, 7.25, -900.0, 1e9, -1e-30, 65504.0, 0.1]):
        x[1, 32 * j + (5 * j) % 32] = v
    # row 2: all zero
    _q8_check(x, x, 3, 256)
    # the same values through the bf16 path (values chosen exactly representable where it matters)
    bits = workloads.f32_to_bf16_bits(x)
    _q8_check(workloads.bf16_bits_to_f32(bits).reshape(3, 256), bits.reshape(3, 256), 3, 256)


def test_q8_1_hand_written_bytes():
    """The GPU quantizer's bytes equal the vector written out by hand (layout and values)."""
    x, want = q8_1_byte_vector()
    out = torch.empty(want.size, dtype=torch.uint8, device=dev())
    lib().q8_1_quantize_act(to_dev(x), out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.array_equal(got, want), f"first mismatch at byte {int(np.argmax(got != want))}"


def test_q8_1_hand_worked_blocks():
    """Hand-worked blocks, including amax exactly 2^-120 (subnormal d) and the float32 below it."""
    blocks = list(q8_1_blocks().values())
    x = np.stack([b["x"] for b in blocks]).reshape(1, -1)
    x = np.concatenate([x, np.zeros((1, (-x.shape[1]) % 256), np.float32)], axis=1)
    k = x.shape[1]
    out = torch.empty(lib().q8_1_bytes(1, k), dtype=torch.uint8, device=dev())
    lib().q8_1_quantize_act(to_dev(x), out)
    torch.cuda.synchronize()
    q, d, s = oracle.q8_1_from_bytes(out.cpu().numpy(), 1, k)
    for i, b in enumerate(blocks):
        assert np.array_equal(q[0, 32 * i:32 * i + 32].astype(np.int64), b["q"]), i
        if "d" in b:
            assert d[0, i] == np.float32(b["d"]) and s[0, i] == np.float32(b["s"]), i
        if "dbits" in b:
            assert int(d[0, i:i + 1].view(np.uint32)[0]) == b["dbits"], i
            assert int(s[0, i:i + 1].view(np.uint32)[0]) == b["sbits"], i


def test_q8_1_random_both_dtypes():
    c = workloads.small_config(1024, 256, 37, "f32", ("channels", 0.01, 1000.0))
    xf, xb = workloads.activations(c)
    _q8_check(xf, xb, 37, 1024)
    c = workloads.small_config(1024, 256, 37, "bf16", ("entries", 0.01, 900.0))
    xf, xb = workloads.activations(c)
    _q8_check(xf, xb, 37, 1024)


@pytest.mark.parametrize("kind", ["gauss", "mixed", "bf16"])
def test_quantize_weights_bit_exact(kind):
    if kind == "gauss":
        w = workloads.normal(21, 1, 96 * 1024).reshape(96, 1024).astype(np.float32)
        buf = w
    elif kind == "mixed":
        u = workloads.normal(22, 1, 64 * 512).reshape(64, 512)
        sc = np.exp(workloads.normal(22, 2, 64 * 16).reshape(64, 16) * 2.0).repeat(32, axis=1)
        w = (u * sc).astype(np.float32)
        w[0] = np.abs(w[0])
        w[1] = -np.abs(w[1])
        w[2, :256] = 0.0
        w[3, 32:64] = 0.0
        buf = w
    else:
        bits = workloads.f32_to_bf16_bits(workloads.normal(23, 1, 32 * 768).astype(np.float32) * 0.02)
        w = workloads.bf16_bits_to_f32(bits).reshape(32, 768)
        buf = bits.reshape(32, 768)
    out = lib().q4k_quantize_weights(to_dev(buf))
    ref = oracle.quantize_q4k(w)
    got = out.cpu().numpy()
    assert np.array_equal(got, ref), f"first mismatch at byte {int(np.argmax(got.reshape(-1) != ref.reshape(-1)))}"
    assert lib().q4k_check_device_error() == 0


def test_quantize_weights_range_error_is_reported():
    w = np.full((2, 256), 1e9, np.float32)
    out = lib().q4k_quantize_weights(to_dev(w))
    assert lib().q4k_check_device_error() == 9          # Q4K_ERR_RANGE
    assert lib().q4k_check_device_error() == 0          # cleared after reading
    assert np.all(out.cpu().numpy() == 0)
