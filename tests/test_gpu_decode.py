"""Parity of the decode path (m <= 8) with the oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import TIGHT_L2, TIGHT_MAX, check_close, dev, guarded_f32, guards_intact, lib, to_dev, torch

pytestmark = pytest.mark.gpu

# The acceptance bounds are 1e-3 (L2-relative and element-wise). The decode
# arithmetic (fp16 hi+lo activations, ~2^-22 relative, exact q*scale, fp32
# accumulation) sits far below them; the TIGHT bounds catch a slip the
# acceptance bounds would hide.


def _run(cfg, x=None, m=None):
    wg, wu, wd = workloads.weights(cfg)
    if x is None:
        x, _ = workloads.activations(cfg, m=m)
    m, H = x.shape
    buf, y = guarded_f32(m * H)
    lib().ffn_q4k_swiglu(to_dev(x), to_dev(wg), to_dev(wu), to_dev(wd), y=y.view(m, H))
    torch.cuda.synchronize()
    assert guards_intact(buf)
    ref, _ = oracle.ffn_decode(x, wg, wu, wd)
    return y.view(m, H).cpu().numpy(), ref


@pytest.mark.parametrize("cfg_index", [0, 1, 2])
def test_decode_workloads(cfg_index):
    y, ref = _run(workloads.CONFIGS[cfg_index])
    check_close(y, ref, TIGHT_L2, TIGHT_MAX, f"config {cfg_index}")
    assert lib().q4k_check_device_error() == 0


@pytest.mark.parametrize("H,I,m", [(256, 256, 1), (256, 512, 2), (512, 256, 3), (768, 1280, 4), (1024, 768, 5),
                                   (2304, 1792, 6), (1280, 3328, 7), (4096, 2048, 8), (256, 4352, 8),
                                   (6912, 512, 1)])
def test_decode_shape_sweep(H, I, m):
    c = workloads.small_config(H, I, m, "f32", ("channels", 0.01, 50.0))
    y, ref = _run(c)
    check_close(y, ref, TIGHT_L2, TIGHT_MAX)


def test_decode_repeatable_and_deterministic():
    c = workloads.small_config(1024, 2816, 8)
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    x, _ = workloads.activations(c)
    xd = to_dev(x)
    y1 = lib().ffn_q4k_swiglu(xd, wg, wu, wd).cpu().numpy()
    y2 = lib().ffn_q4k_swiglu(xd, wg, wu, wd).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_decode_repeated_calls_on_the_same_buffers():
    """A decode loop calls with the same buffers every token; such repeats are replayed
    from a recorded launch sequence, which must read the current x every time."""
    c = workloads.small_config(1024, 2816, 2)
    wg, wu, wd = workloads.weights(c)
    dg, du, dd = to_dev(wg), to_dev(wu), to_dev(wd)
    xd = torch.empty((2, 1024), dtype=torch.float32, device=dev())
    y = torch.empty((2, 1024), dtype=torch.float32, device=dev())
    outs = []
    for k in range(4):
        x, _ = workloads.activations(c, seed=c.seed + 17 * k)
        xd.copy_(torch.from_numpy(x))
        lib().ffn_q4k_swiglu(xd, dg, du, dd, y=y)
        torch.cuda.synchronize()
        ref, _ = oracle.ffn_decode(x, wg, wu, wd)
        check_close(y.cpu().numpy(), ref, TIGHT_L2, TIGHT_MAX, f"call {k}")
        outs.append(y.cpu().numpy().copy())
    x, _ = workloads.activations(c, seed=c.seed)  # the first input again: the same bits
    xd.copy_(torch.from_numpy(x))
    lib().ffn_q4k_swiglu(xd, dg, du, dd, y=y)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), outs[0].view(np.uint32))
    assert lib().q4k_check_device_error() == 0


def test_decode_special_inputs():
    c = workloads.small_config(512, 768, 3)
    wg, wu, wd = workloads.weights(c)
    # zero input -> exactly zero output
    y = lib().ffn_q4k_swiglu(to_dev(np.zeros((3, 512), np.float32)), to_dev(wg), to_dev(wu), to_dev(wd))
    assert np.all(y.cpu().numpy() == 0)
    # huge and tiny activations in one token (exercise the per-superblock exponent)
    x = np.zeros((3, 512), np.float32)
    x[0] = workloads.normal(5, 1, 512) * 1e4
    x[1] = workloads.normal(5, 2, 512) * 1e-6
    x[2, ::7] = 3.0e5
    y, ref = _run(c, x=x)
    check_close(y, ref, TIGHT_L2, TIGHT_MAX)


@pytest.mark.parametrize("row", [0, 1, 2])
def test_decode_one_token_extreme_inputs(row):
    """One token (the block-diagonal path and its SwiGLU): activations that drive the gate to
    magnitudes in the 1e5 range (silu's both tails), to 1e-6, and sparse spikes."""
    c = workloads.small_config(512, 768, 1)
    x = np.zeros((1, 512), np.float32)
    if row == 0:
        x[0] = workloads.normal(5, 1, 512) * 1e4
    elif row == 1:
        x[0] = workloads.normal(5, 2, 512) * 1e-6
    else:
        x[0, ::7] = 3.0e5
    y, ref = _run(c, x=x)
    assert np.all(np.isfinite(y))
    check_close(y, ref, TIGHT_L2, TIGHT_MAX, f"one token, input {row}")


@pytest.mark.parametrize("H,I,m", [(16384, 256, 1), (16384, 256, 3), (256, 32768, 2)])
def test_decode_many_k_chunks(H, I, m):
    """Shapes the planner splits into 8 gate/up K-chunks (hidden 16384, one or three tokens) or
    16 down K-chunks (inter 32768): the chunk sums take their loads in batches (4 chunks in the
    SwiGLU kernel, 8 in the down-chunk sum), and every batch boundary is crossed."""
    c = workloads.small_config(H, I, m, "f32", ("channels", 0.01, 20.0))
    y, ref = _run(c)
    check_close(y, ref, TIGHT_L2, TIGHT_MAX, f"h {H} i {I} m {m}")


@pytest.mark.parametrize("m", [1, 4])
def test_decode_bf16_input_through_ex(m):
    """bf16 activations: one token (x's fragments built inside the gate/up GEMV) and four."""
    c = workloads.small_config(768, 1024, m, "bf16", ("channels", 0.01, 100.0))
    wg, wu, wd = workloads.weights(c)
    xf, xb = workloads.activations(c)
    ws = torch.zeros(lib().ffn_q4k_workspace_bytes(m, 768, 1024), dtype=torch.uint8, device=dev())
    y = lib().ffn_q4k_swiglu_ex(to_dev(xb), to_dev(wg), to_dev(wu), to_dev(wd), ws)
    ref, _ = oracle.ffn_decode(xf, wg, wu, wd)
    check_close(y.cpu().numpy(), ref, TIGHT_L2, TIGHT_MAX)


def test_workspace_too_small_is_rejected():
    c = workloads.small_config(256, 512, 1)
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    x = to_dev(np.ones((1, 256), np.float32))
    need = lib().ffn_q4k_workspace_bytes(1, 256, 512)
    ws = torch.zeros(need - 256, dtype=torch.uint8, device=dev())
    with pytest.raises(lib().Q4KError) as e:
        lib().ffn_q4k_swiglu_ex(x, wg, wu, wd, ws)
    assert e.value.status == 8


@pytest.mark.parametrize("m", [9, 16, 17, 23, 24])
def test_decode_passes_of_16_tokens(m):
    """9-24 tokens run as decode passes of at most 16 tokens (float32 activations): each pass's
    rows equal the call on those tokens alone, and the whole output meets the fp64 oracle."""
    c = workloads.small_config(1024, 1536, m, "f32", ("channels", 0.01, 50.0))
    wg, wu, wd = workloads.weights(c)
    dg, du, dd = to_dev(wg), to_dev(wu), to_dev(wd)
    x, _ = workloads.activations(c)
    y = lib().ffn_q4k_swiglu(to_dev(x), dg, du, dd).cpu().numpy()
    for t0 in range(0, m, 16):
        ys = lib().ffn_q4k_swiglu(to_dev(x[t0:t0 + 16]), dg, du, dd).cpu().numpy()
        assert np.array_equal(y[t0:t0 + 16].view(np.uint32), ys.view(np.uint32))
    ref, _ = oracle.ffn_decode(x, wg, wu, wd)
    check_close(y, ref, TIGHT_L2, TIGHT_MAX)
    assert lib().ffn_q4k_workspace_h_q8_1_offset(m, 1024, 1536) == 0


def test_binding_enqueues_on_the_current_stream():
    """Without a stream argument the binding uses PyTorch's current stream of the current device."""
    q = lib()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert q._stream(None) == s.cuda_stream == torch.cuda.current_stream().cuda_stream
    assert q._stream(None) == torch.cuda.current_stream().cuda_stream
    assert q._stream(s) == s.cuda_stream
