"""Parity of the prefill path (m >= 25: Q8_1 activations, tcgen05 Q4_K x Q8_1 GEMM) with the oracle."""
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


def _run(cfg, m=None, sample=None):
    wg, wu, wd = workloads.weights(cfg)
    xf, xb = workloads.activations(cfg, m=m)
    m, H = xf.shape
    I = cfg.inter
    need = lib().ffn_q4k_workspace_bytes(m, H, I)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev())
    buf, y = guarded_f32(m * H)
    lib().ffn_q4k_swiglu_ex(to_dev(xb), to_dev(wg), to_dev(wu), to_dev(wd), ws, y=y.view(m, H))
    torch.cuda.synchronize()
    assert guards_intact(buf)
    assert lib().q4k_check_device_error() == 0
    y = y.view(m, H).cpu().numpy()
    off = lib().ffn_q4k_workspace_h_q8_1_offset(m, H, I)
    hq_gpu = oracle.q8_1_from_bytes(ws[off:off + lib().q8_1_bytes(m, I)].cpu().numpy(), m, I)
    rows = np.arange(m) if sample is None else sample
    ref = oracle.ffn_prefill(xf[rows], wg, wu, wd)
    return y[rows], ref, tuple(a[rows] for a in hq_gpu), wd


def _check(y, ref, hq_gpu, wd):
    err, _ = check_close(y, ref["y"], ACCEPT_L2, ACCEPT_MAX)
    hq, hd, hs = ref["hq"]
    gq, gd, gs = hq_gpu
    flips = np.count_nonzero(gq != hq)
    assert flips <= HQ_FLIP_FRAC * hq.size, flips
    # A flip moves a value by one quant step of its block. Where g or u nearly
    # cancels, the float32 accumulation error (~1e-7 of sum|w*x|) can be a large
    # part of h itself, so a handful of values (and the scale of their block,
    # when such a value is the block maximum) may move further; they must stay rare.
    dv = np.abs(oracle.dequantize_q8_1(gq, gd) - oracle.dequantize_q8_1(hq, hd))
    step = np.repeat(np.maximum(gd, hd).astype(np.float64), 32, axis=1)
    far = np.count_nonzero(dv > 1.01 * step + 1e-30 * 127)
    assert far <= max(1, HQ_FAR_FRAC * hq.size), far
    # the down GEMM alone, fed the GPU's own Q8_1(h)
    y_down = oracle.ffn_down_from_q8_1(gq, gd, wd)
    check_close(y, y_down, DOWN_TIGHT, TIGHT_MAX, "down stage on the GPU's Q8_1(h)")
    return err


@pytest.mark.parametrize("H,I,m", [(256, 256, 25), (256, 512, 48), (512, 256, 127), (256, 768, 128),
                                   (768, 512, 129), (1024, 1280, 200), (512, 2048, 257), (1280, 256, 64)])
def test_prefill_shape_sweep(H, I, m):
    c = workloads.small_config(H, I, m, "bf16", ("channels", 0.01, 100.0))
    y, ref, hq, wd = _run(c)
    _check(y, ref, hq, wd)


def test_prefill_float32_input():
    c = workloads.small_config(512, 768, 33, "f32", ("entries", 0.001, 900.0))
    y, ref, hq, wd = _run(c)
    _check(y, ref, hq, wd)


def test_prefill_config3_full():
    y, ref, hq, wd = _run(workloads.CONFIGS[3])
    _check(y, ref, hq, wd)


def test_prefill_config4_full():
    """The 27B-shaped long prefill (2048 tokens) in the benchmark's launch configuration,
    every token checked: the persistent tile walk, the down projection's K-split tail and
    every token-tile edge depend on the token index."""
    y, ref, hq, wd = _run(workloads.CONFIGS[4])
    _check(y, ref, hq, wd)


def test_prefill_zero_input():
    c = workloads.small_config(256, 512, 40, "bf16")
    wg, wu, wd = workloads.weights(c)
    ws = torch.zeros(lib().ffn_q4k_workspace_bytes(40, 256, 512), dtype=torch.uint8, device=dev())
    x = torch.zeros((40, 256), dtype=torch.bfloat16, device=dev())
    y = lib().ffn_q4k_swiglu_ex(x, to_dev(wg), to_dev(wu), to_dev(wd), ws)
    assert torch.count_nonzero(y).item() == 0


def test_prefill_repeatable():
    c = workloads.small_config(512, 1024, 140, "bf16", ("channels", 0.01, 100.0))
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    _, xb = workloads.activations(c)
    xd = to_dev(xb)
    ws = torch.zeros(lib().ffn_q4k_workspace_bytes(140, 512, 1024), dtype=torch.uint8, device=dev())
    y1 = lib().ffn_q4k_swiglu_ex(xd, wg, wu, wd, ws).cpu().numpy()
    y2 = lib().ffn_q4k_swiglu_ex(xd, wg, wu, wd, ws).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("H", [43520, 43776])
def test_prefill_widest_hidden_sizes(H):
    """x's row is quantized and expanded by one kernel up to hidden 43520 (its quants and block
    scales held in shared memory) and by two kernels above that; both sides of the boundary."""
    c = workloads.small_config(H, 256, 25, "bf16", ("channels", 0.01, 100.0))
    y, ref, hq, wd = _run(c)
    _check(y, ref, hq, wd)


@pytest.mark.parametrize("H,I,m", [(2048, 10240, 32), (1024, 10240, 200)])
def test_prefill_gate_up_tail_split(H, I, m):
    """More gate/up tiles than SMs with a short last round (160 and 320 tiles of 64 inter rows on
    152 SMs): the last round's tiles are split along K, and their SwiGLU and Q8_1 follow the sum
    of the slices in a separate kernel."""
    c = workloads.small_config(H, I, m, "bf16", ("channels", 0.01, 100.0))
    y, ref, hq, wd = _run(c)
    _check(y, ref, hq, wd)
