"""The FP8 tensor-core Q4_K x Q8_1 GEMM (tcgen05 kind::f8f6f4) against the oracle.

Every integer product is exact on this path (4-bit quants and the two 4-bit halves of
each Q8_1 quant are exact E4M3 values); the scales are applied in float32 per 32-weight
sub-block. So the result must match the fp64 oracle's product of the dequantized
operands to float32 accumulation error."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import TIGHT_L2, TIGHT_MAX, check_close, dev, lib, to_dev, torch

pytestmark = pytest.mark.gpu


def _gemm(x, blocks):
    m, k = x.shape
    n = blocks.shape[0]
    xq8 = torch.empty(lib().q8_1_bytes(m, k), dtype=torch.uint8, device=dev())
    lib().q8_1_quantize_act(to_dev(x), xq8)
    out = torch.full((m, n), float("nan"), dtype=torch.float32, device=dev())
    lib().q4k_mmq_fp8(xq8, m, k, to_dev(blocks), out=out)
    torch.cuda.synchronize()
    assert lib().q4k_check_device_error() == 0
    q, d, _ = oracle.quantize_q8_1(x)
    ref = oracle.dequantize_q8_1(q, d) @ oracle.dequantize_q4k(blocks).T
    return out.cpu().numpy(), ref


@pytest.mark.parametrize("m,k,n", [(1, 256, 128), (37, 512, 256), (128, 768, 128), (200, 1280, 384),
                                   (129, 4096, 256)])
def test_fp8_gemm_matches_oracle(m, k, n):
    c = workloads.small_config(k, n, m, "f32", ("channels", 0.01, 40.0))
    x, _ = workloads.activations(c)
    blocks = workloads.q4k_blocks(c.seed, 3, n, k)
    y, ref = _gemm(x, blocks)
    check_close(y, ref, TIGHT_L2, TIGHT_MAX)


def test_fp8_gemm_gate_projection_27b_sampled():
    """The 27B-shaped gate projection (2048 tokens, k = 5120) over 1024 of its 17408 rows."""
    cfg = workloads.LONG_PREFILL_27B
    xf, _ = workloads.activations(cfg)
    wg = workloads.weights(cfg)[0][:1024]
    y, ref = _gemm(xf, wg)
    check_close(y, ref, TIGHT_L2, TIGHT_MAX)


def test_fp8_gemm_one_hot_rows_gather_q8_values():
    """One-hot rows (d = 1, scale 1, min 0, q = 1 at one input) gather the dequantized Q8_1 values."""
    m, k, n = 64, 512, 128
    rng = np.random.default_rng(8)
    blocks = np.zeros((n, k // 256, 144), np.uint8)
    blocks[:, :, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    sc = np.ones((n, k // 256, 8), np.int64)
    blocks[:, :, 4:16] = oracle.pack_scales_mins(sc, np.zeros_like(sc))
    cols = rng.integers(0, k, n)
    for r, c in enumerate(cols):
        sb, i = divmod(int(c), 256)
        g, w = divmod(i, 64)
        byte = 16 + 32 * g + (w % 32)
        blocks[r, sb, byte] |= 1 if w < 32 else 16
    x = (rng.standard_normal((m, k)) * 3).astype(np.float32)
    y, ref = _gemm(x, blocks)
    q, d, _ = oracle.quantize_q8_1(x)
    hand = oracle.dequantize_q8_1(q, d)[:, cols]
    check_close(ref, hand, 1e-12, 1e-12, "oracle gather")
    check_close(y, hand, 1e-6, 1e-6, "gather")


def test_fp8_gemm_rejects_bad_shapes():
    q = lib()
    A = torch.zeros(1 << 16, dtype=torch.uint8, device=dev())
    W = torch.zeros((100, 1, 144), dtype=torch.uint8, device=dev())   # n not a multiple of 128
    with pytest.raises(q.Q4KError) as e:
        q.q4k_mmq_fp8(A, 4, 256, W, workspace=A, out=torch.zeros(400, device=dev()))
    assert e.value.status == 2
    assert q.q4k_mmq_fp8_workspace_bytes(4, 300) == 0
