"""x and y in page-locked host memory (read and written by the kernels across the host link)
give the same bits as device buffers; host memory the device cannot address is refused."""
import numpy as np
import pytest

import workloads
from tests.gpu_util import dev, lib, to_dev, torch

pytestmark = pytest.mark.gpu


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def _same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint32), np.asarray(b).view(np.uint32))


@pytest.mark.parametrize("m", [1, 8])
def test_decode_host_io(m):
    c = workloads.small_config(1024, 2816, m)
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    x, _ = workloads.activations(c)
    y_dev = lib().ffn_q4k_swiglu(to_dev(x), wg, wu, wd).cpu().numpy()
    xh = _pinned(x)
    yh = torch.empty((m, 1024), dtype=torch.float32).pin_memory()
    for _ in range(2):  # the second call replays the recorded launch sequence
        yh.fill_(float("nan"))
        lib().ffn_q4k_swiglu(xh, wg, wu, wd, y=yh)
        torch.cuda.synchronize()
        assert _same(yh.numpy(), y_dev)


def test_q8_1_decode_and_prefill_host_io():
    for m, dt in [(1, "f32"), (24, "bf16")]:
        c = workloads.small_config(512, 768, m, dt)
        wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
        _, xb = workloads.activations(c)
        ws = torch.zeros(lib().ffn_q4k_q8_1_workspace_bytes(m, 512, 768), dtype=torch.uint8, device=dev())
        y_dev = lib().ffn_q4k_swiglu_q8_1(to_dev(xb), wg, wu, wd, ws).cpu().numpy()
        xh = to_dev(xb).cpu().pin_memory()
        yh = torch.empty((m, 512), dtype=torch.float32).pin_memory()
        lib().ffn_q4k_swiglu_q8_1(xh, wg, wu, wd, ws, y=yh)
        torch.cuda.synchronize()
        assert _same(yh.numpy(), y_dev)


def test_q6k_host_io():
    blocks = to_dev(workloads.q6k_blocks(3, 1, 256, 1024))
    x = workloads.normal(3, 4, 2 * 1024).reshape(2, 1024).astype(np.float32)
    ws = torch.empty(lib().q6k_gemv_workspace_bytes(2, 256, 1024), dtype=torch.uint8, device=dev())
    y_dev = lib().q6k_gemv(to_dev(x), blocks, ws).cpu().numpy()
    yh = torch.empty((2, 256), dtype=torch.float32).pin_memory()
    lib().q6k_gemv(_pinned(x), blocks, ws, y=yh)
    torch.cuda.synchronize()
    assert _same(yh.numpy(), y_dev)


def test_pageable_host_memory_is_refused():
    c = workloads.small_config(256, 512, 1)
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    x = torch.zeros((1, 256), dtype=torch.float32)  # pageable: not pinned
    assert not x.is_pinned()
    with pytest.raises(lib().Q4KError) as e:
        lib().ffn_q4k_swiglu(x, wg, wu, wd, y=torch.empty((1, 256), dtype=torch.float32, device=dev()))
    assert e.value.status == 10
