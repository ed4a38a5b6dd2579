"""Parity of the decode path with Q8_1 activations (m <= 8, integer dot products) with the oracle.

The oracle is the same Q8_1 pipeline the prefill path follows (x -> Q8_1, fp64 gate/up over the
dequantized operands, h rounded to float32 and re-quantized to Q8_1, fp64 down), so the bar is
the prefill one: the whole output within the acceptance bound, Q8_1(h) equal to the oracle's
except where h sits on a rounding boundary, and the down projection alone (fed the GPU's own
Q8_1(h)) within float32 rounding of the fp64 result.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import (ACCEPT_L2, ACCEPT_MAX, TIGHT_MAX, check_close, dev, guarded_f32, guards_intact, lib,
                            to_dev, torch)

pytestmark = pytest.mark.gpu

DOWN_TIGHT = 1e-5      # y against the oracle's down stage fed the GPU's own Q8_1(h), L2-relative
HQ_FLIP_FRAC = 2e-3    # Q8_1(h) bytes may differ where h sits on a rounding boundary
HQ_FAR_FRAC = 1e-4     # ... or, rarely, by more than one step where g or u nearly cancels


def _run(cfg, x=None, m=None, bf16=False):
    wg, wu, wd = workloads.weights(cfg)
    if x is None:
        xf, xb = workloads.activations(cfg, m=m)
        x_in = xb if bf16 else xf
        x = xf
    else:
        x_in = x
    m, H = x.shape
    I = cfg.inter
    ws = torch.full((lib().ffn_q4k_q8_1_workspace_bytes(m, H, I),), 0xA5, dtype=torch.uint8, device=dev())
    buf, y = guarded_f32(m * H)
    lib().ffn_q4k_swiglu_q8_1(to_dev(x_in), to_dev(wg), to_dev(wu), to_dev(wd), ws, y=y.view(m, H))
    torch.cuda.synchronize()
    assert guards_intact(buf)
    assert lib().q4k_check_device_error() == 0
    off = lib().ffn_q4k_q8_1_workspace_h_offset(m, H, I)
    hq_gpu = oracle.q8_1_from_bytes(ws[off:off + lib().q8_1_bytes(m, I)].cpu().numpy(), m, I)
    ref = oracle.ffn_prefill(x, wg, wu, wd)
    return y.view(m, H).cpu().numpy(), ref, hq_gpu, wd


def _check(y, ref, hq_gpu, wd):
    err, _ = check_close(y, ref["y"], ACCEPT_L2, ACCEPT_MAX)
    hq, hd, _ = ref["hq"]
    gq, gd, gs = hq_gpu
    flips = np.count_nonzero(gq != hq)
    assert flips <= max(1, HQ_FLIP_FRAC * hq.size), flips
    dv = np.abs(oracle.dequantize_q8_1(gq, gd) - oracle.dequantize_q8_1(hq, hd))
    step = np.repeat(np.maximum(gd, hd).astype(np.float64), 32, axis=1)
    far = np.count_nonzero(dv > 1.01 * step)
    assert far <= max(1, HQ_FAR_FRAC * hq.size), far
    # the GPU's Q8_1(h) is a valid Q8_1 encoding of itself: s = d * sum(q) in float32
    sums = gq.reshape(gq.shape[0], -1, 32).astype(np.int64).sum(axis=2).astype(np.float32)
    assert np.array_equal(gs, (gd * sums).astype(np.float32))
    # the down GEMV alone, fed the GPU's own Q8_1(h)
    check_close(y, oracle.ffn_down_from_q8_1(gq, gd, wd), DOWN_TIGHT, TIGHT_MAX, "down stage on the GPU's Q8_1(h)")
    return err


@pytest.mark.parametrize("cfg_index", [0, 1, 2])
def test_decode_q8_workloads(cfg_index):
    """The three decode workloads (tiny, LLaMA-7B m = 1, 13B m = 8 with outlier channels)."""
    _check(*_run(workloads.CONFIGS[cfg_index]))


@pytest.mark.parametrize("H,I,m", [(256, 256, 1), (256, 512, 2), (512, 256, 3), (768, 1280, 4), (1024, 768, 5),
                                   (2304, 1792, 6), (1280, 3328, 7), (4096, 2048, 8), (256, 4352, 8),
                                   (6912, 512, 1), (512, 6912, 2)])
def test_decode_q8_shape_sweep(H, I, m):
    """Every token-count kernel (1, 2, 4, 8 tokens, with padding tokens), ragged K-chunks and row units."""
    c = workloads.small_config(H, I, m, "f32", ("channels", 0.01, 50.0))
    _check(*_run(c))


@pytest.mark.parametrize("m", [1, 2, 3])
def test_decode_q8_bf16_input(m):
    """bf16 activations: 1-2 tokens (x quantized inside the gate/up GEMV) and 3 (the float32
    path's kernels)."""
    c = workloads.small_config(1024, 1536, m, "bf16", ("entries", 0.001, 900.0))
    _check(*_run(c, bf16=True))


def test_decode_q8_zero_input():
    """x = 0 quantizes to zero blocks (d = s = 0), so h = 0 and y = 0 exactly."""
    c = workloads.small_config(512, 768, 2)
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    ws = torch.empty(lib().ffn_q4k_q8_1_workspace_bytes(2, 512, 768), dtype=torch.uint8, device=dev())
    x = torch.zeros((2, 512), dtype=torch.float32, device=dev())
    y = lib().ffn_q4k_swiglu_q8_1(x, wg, wu, wd, ws)
    assert torch.count_nonzero(y).item() == 0


def test_decode_q8_one_hot_weights():
    """One-hot weights (d = 1, scales 1, mins 0, a single quant 1 per row): every GEMV is a
    gather, so the result follows by hand from the Q8_1 values, h = silu(x8[src_g]) * x8[src_u]
    and y = Q8(h)[src_d]."""
    H, I, m = 512, 768, 2
    rng = np.random.default_rng(11)

    def one_hot(rows, cols):
        blocks = np.zeros((rows, cols // 256, 144), dtype=np.uint8)
        blocks[:, :, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), dtype=np.uint8)  # d = 1, dmin = 0
        blocks[:, :, 4:8] = 1     # sub-blocks 0-3: scale 1 (their mins, bytes 8-11, stay 0)
        blocks[:, :, 12:16] = 1   # sub-blocks 4-7: scale low nibble 1, min nibble 0
        src = rng.integers(0, cols, size=rows)
        for r, c in enumerate(src):
            b, w = divmod(int(c), 256)
            grp, pos = divmod(w, 64)
            blocks[r, b, 16 + 32 * grp + pos % 32] = 1 if pos < 32 else 16
        return blocks, src

    wg, sg = one_hot(I, H)
    wu, su = one_hot(I, H)
    wd, sd = one_hot(H, I)
    onehot = np.zeros((I, H))
    onehot[np.arange(I), sg] = 1.0
    assert np.array_equal(oracle.dequantize_q4k(wg), onehot)
    x = rng.standard_normal((m, H)).astype(np.float32)
    xq, xd, _ = oracle.quantize_q8_1(x)
    x8 = oracle.dequantize_q8_1(xq, xd)
    h = ((x8[:, sg] / (1.0 + np.exp(-x8[:, sg]))) * x8[:, su]).astype(np.float32)
    hq, hd, _ = oracle.quantize_q8_1(h)
    y_hand = oracle.dequantize_q8_1(hq, hd)[:, sd]
    ws = torch.empty(lib().ffn_q4k_q8_1_workspace_bytes(m, H, I), dtype=torch.uint8, device=dev())
    y = lib().ffn_q4k_swiglu_q8_1(to_dev(x), to_dev(wg), to_dev(wu), to_dev(wd), ws).cpu().numpy()
    off = lib().ffn_q4k_q8_1_workspace_h_offset(m, H, I)
    gq, gd, _ = oracle.q8_1_from_bytes(ws[off:off + lib().q8_1_bytes(m, I)].cpu().numpy(), m, I)
    # gate/up: float32 silu may move an h that sits on a rounding boundary by one step
    assert np.count_nonzero(gq != hq) <= 2
    assert np.all(np.abs(gq.astype(int) - hq.astype(int)) <= 1)
    # down: a gather of the GPU's own Q8_1(h), exact up to the float32 product d8 * q8
    check_close(y, oracle.dequantize_q8_1(gq, gd)[:, sd], 1e-6, 1e-6, "gather of the GPU's Q8_1(h)")
    check_close(y, y_hand, ACCEPT_L2, ACCEPT_MAX, "hand-computed gather")


def test_decode_q8_repeated_calls_on_the_same_buffers():
    """Repeats with the same buffers replay a recorded launch sequence that must read the current x."""
    c = workloads.small_config(1024, 2816, 1)
    wg, wu, wd = workloads.weights(c)
    dg, du, dd = to_dev(wg), to_dev(wu), to_dev(wd)
    xd = torch.empty((1, 1024), dtype=torch.float32, device=dev())
    y = torch.empty((1, 1024), dtype=torch.float32, device=dev())
    ws = torch.empty(lib().ffn_q4k_q8_1_workspace_bytes(1, 1024, 2816), dtype=torch.uint8, device=dev())
    outs = []
    for k in range(4):
        x, _ = workloads.activations(c, seed=c.seed + 17 * k)
        xd.copy_(torch.from_numpy(x))
        lib().ffn_q4k_swiglu_q8_1(xd, dg, du, dd, ws, y=y)
        torch.cuda.synchronize()
        check_close(y.cpu().numpy(), oracle.ffn_prefill(x, wg, wu, wd)["y"], ACCEPT_L2, ACCEPT_MAX, f"call {k}")
        outs.append(y.cpu().numpy().copy())
    x, _ = workloads.activations(c, seed=c.seed)
    xd.copy_(torch.from_numpy(x))
    lib().ffn_q4k_swiglu_q8_1(xd, dg, du, dd, ws, y=y)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), outs[0].view(np.uint32))


@pytest.mark.parametrize("m", [9, 20, 24])
def test_decode_q8_passes_of_16_tokens(m):
    """9-24 tokens run as decode passes of at most 16 tokens: each pass's rows equal the call on
    those tokens alone, and the whole output meets the Q8_1 oracle."""
    c = workloads.small_config(1024, 1536, m, "f32", ("channels", 0.01, 50.0))
    wg, wu, wd = workloads.weights(c)
    dg, du, dd = to_dev(wg), to_dev(wu), to_dev(wd)
    x, _ = workloads.activations(c)
    ws = torch.empty(lib().ffn_q4k_q8_1_workspace_bytes(m, 1024, 1536), dtype=torch.uint8, device=dev())
    y = lib().ffn_q4k_swiglu_q8_1(to_dev(x), dg, du, dd, ws).cpu().numpy()
    for t0 in range(0, m, 16):
        xs = x[t0:t0 + 16]
        w1 = torch.empty(lib().ffn_q4k_q8_1_workspace_bytes(len(xs), 1024, 1536), dtype=torch.uint8, device=dev())
        ys = lib().ffn_q4k_swiglu_q8_1(to_dev(xs), dg, du, dd, w1).cpu().numpy()
        assert np.array_equal(y[t0:t0 + 16].view(np.uint32), ys.view(np.uint32))
    check_close(y, oracle.ffn_prefill(x, wg, wu, wd)["y"], ACCEPT_L2, ACCEPT_MAX)
    assert lib().ffn_q4k_q8_1_workspace_h_offset(m, 1024, 1536) == 0


def test_q8_1_entry_point_at_prefill_sizes_is_the_prefill_path():
    """For m >= 25 the Q8_1 entry point and ffn_q4k_swiglu_ex compute the same bytes."""
    c = workloads.small_config(512, 768, 48, "bf16", ("channels", 0.01, 100.0))
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    _, xb = workloads.activations(c)
    xd = to_dev(xb)
    ws1 = torch.zeros(lib().ffn_q4k_q8_1_workspace_bytes(48, 512, 768), dtype=torch.uint8, device=dev())
    ws2 = torch.zeros(lib().ffn_q4k_workspace_bytes(48, 512, 768), dtype=torch.uint8, device=dev())
    y1 = lib().ffn_q4k_swiglu_q8_1(xd, wg, wu, wd, ws1).cpu().numpy()
    y2 = lib().ffn_q4k_swiglu_ex(xd, wg, wu, wd, ws2).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_decode_q8_rejects_bad_arguments():
    c = workloads.small_config(256, 512, 1)
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    x = torch.zeros((1, 256), dtype=torch.float32, device=dev())
    need = lib().ffn_q4k_q8_1_workspace_bytes(1, 256, 512)
    small = torch.empty(need - 256, dtype=torch.uint8, device=dev())
    with pytest.raises(lib().Q4KError) as e:
        lib().ffn_q4k_swiglu_q8_1(x, wg, wu, wd, small)
    assert e.value.status == 8
    assert lib().ffn_q4k_q8_1_workspace_bytes(1, 300, 512) == 0
