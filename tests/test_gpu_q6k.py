"""Parity of the Q6_K GEMV (the LM head) with the oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import TIGHT_L2, TIGHT_MAX, check_close, dev, guarded_f32, guards_intact, lib, to_dev, torch

pytestmark = pytest.mark.gpu

# x carried as fp16 hi + lo (about 22 bits), exact weights, fp32 sums: the TIGHT bounds


def _gemv(x_in, blocks, m, n, k):
    ws = torch.empty(lib().q6k_gemv_workspace_bytes(m, n, k), dtype=torch.uint8, device=dev())
    buf, y = guarded_f32(m * n)
    lib().q6k_gemv(to_dev(x_in), to_dev(blocks), ws, y=y.view(m, n))
    torch.cuda.synchronize()
    assert guards_intact(buf)
    assert lib().q4k_check_device_error() == 0
    return y.view(m, n).cpu().numpy()


def test_q6k_dequantize_bit_exact():
    blocks = workloads.q6k_blocks(21, 1, 48, 1280)
    w = lib().q6k_dequantize(to_dev(blocks), 48, 1280).cpu().numpy()
    ref = oracle.dequantize_q6k(blocks).astype(np.float32)
    # every value exact; a zero weight may carry either sign (scale * 0 or 0 * (q - 32))
    assert np.array_equal(w, ref)
    nz = ref != 0
    assert np.array_equal(w[nz].view(np.uint32), ref[nz].view(np.uint32))


def test_q6k_lmhead_tiny():
    c = workloads.LMHEADS[0]
    blocks, x = workloads.lmhead_weights(c), workloads.lmhead_x(c)
    y = _gemv(x, blocks, c.m, c.n, c.k)
    check_close(y, oracle.gemv_q6k(x, blocks), TIGHT_L2, TIGHT_MAX)


def test_q6k_lmhead_llama7b_sampled_rows():
    """The full 32000 x 4096 LM head in the benchmark's launch configuration; 640 rows checked."""
    c = workloads.LMHEADS[1]
    blocks, x = workloads.lmhead_weights(c), workloads.lmhead_x(c)
    y = _gemv(x, blocks, c.m, c.n, c.k)
    rng = np.random.default_rng(6)
    rows = np.sort(np.concatenate([[0, 15, 16, c.n - 1], rng.choice(c.n, 636, replace=False)]))
    ref = oracle.gemv_q6k(x, blocks[rows])
    check_close(y[:, rows], ref, TIGHT_L2, TIGHT_MAX)
    assert np.isfinite(y).all()


@pytest.mark.parametrize("m,n,k", [(1, 16, 256), (2, 48, 512), (3, 64, 1280), (4, 32, 2304), (5, 80, 4096),
                                   (8, 16, 256), (1, 4096, 5120), (6, 96, 8192), (1, 2000 * 16, 1024)])
def test_q6k_shape_sweep(m, n, k):
    """Token tiles of 4 (1-8 tokens), superblock counts odd and even, 2-byte block offsets,
    B fragments held in registers (k <= 4096) or re-read per tile (k > 4096), one and two CTAs per SM."""
    blocks = workloads.q6k_blocks(31 + m, 1, n, k)
    x = workloads.normal(31 + m, 4, m * k).reshape(m, k).astype(np.float32)
    x[:, :: max(1, k // 7)] *= 40.0   # a few large channels
    y = _gemv(x, blocks, m, n, k)
    check_close(y, oracle.gemv_q6k(x, blocks), TIGHT_L2, TIGHT_MAX)


def test_q6k_bf16_input_one_hot_is_exact():
    """One-hot rows (d = 1, scales 1, q = 33 at one input, 32 elsewhere) gather x exactly when
    x is bf16 (its 8 significant bits survive the fp16 hi part)."""
    n, k, m = 64, 768, 3
    rng = np.random.default_rng(4)
    blocks = np.zeros((n, k // 256, 210), dtype=np.uint8)
    blocks[..., 128:192] = 0xAA
    blocks[..., 192:208] = 1
    blocks[..., 208:210] = np.frombuffer(np.float16(1.0).tobytes(), dtype=np.uint8)
    src = rng.integers(0, k, size=n)
    for r, c in enumerate(src):
        b, i = divmod(int(c), 256)
        h, rr = divmod(i, 128)
        s, l = divmod(rr, 32)
        blocks[r, b, 64 * h + l + 32 * (s % 2)] |= 1 if s < 2 else 0x10
    xf = rng.standard_normal((m, k)).astype(np.float32)
    bits = workloads.f32_to_bf16_bits(xf)
    xb = workloads.bf16_bits_to_f32(bits).reshape(m, k)
    y = _gemv(bits.reshape(m, k), blocks, m, n, k)
    assert np.array_equal(y, xb[:, src])


def test_q6k_zero_input_and_repeat():
    blocks = workloads.q6k_blocks(41, 1, 256, 1024)
    y = _gemv(np.zeros((2, 1024), dtype=np.float32), blocks, 2, 256, 1024)
    assert np.count_nonzero(y) == 0
    x = workloads.normal(41, 4, 2 * 1024).reshape(2, 1024).astype(np.float32)
    y1, y2 = _gemv(x, blocks, 2, 256, 1024), _gemv(x, blocks, 2, 256, 1024)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_q6k_rejects_bad_shapes():
    blocks = to_dev(workloads.q6k_blocks(1, 1, 32, 256))
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev())
    for m, k in [(9, 256), (1, 300)]:
        x = torch.zeros((m, k), dtype=torch.float32, device=dev())
        with pytest.raises(lib().Q4KError) as e:
            lib().q6k_gemv(x, blocks, ws)
        assert e.value.status == 2
    assert lib().q6k_gemv_workspace_bytes(1, 24, 256) == 0      # n not a multiple of 16
    assert lib().q6k_gemv_workspace_bytes(1, 32, 8448) == 0     # k above 8192
    assert lib().q6k_weight_bytes(32000, 4096) == 32000 * 16 * 210
