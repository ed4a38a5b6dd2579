"""The allocation-free decode entry point against the oracle.

ffn_q4k_swiglu_noalloc serves callers that cannot call cudaMalloc (a server
whose pool owns all device memory, a loop that cannot take cudaMalloc's
device-wide synchronisation): it runs the decode kernels on a static scratch
array inside the library. Two calls in a row must both meet the fp64 oracle
(the scratch keeps the previous call's contents), and agree bit for bit with
ffn_q4k_swiglu, which runs the same kernels on its own workspace. This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes alone.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import TIGHT_L2, TIGHT_MAX, check_close, dev, lib, to_dev, torch

pytestmark = pytest.mark.gpu


def _noalloc():
    f = lib().lib.ffn_q4k_swiglu_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + [ctypes.c_void_p] * 5
    return f


@pytest.mark.parametrize("cfg_index", [1, 2])
def test_noalloc_matches_the_oracle_twice(cfg_index):
    cfg = workloads.CONFIGS[cfg_index]
    wg_h, wu_h, wd_h = workloads.weights(cfg)
    x_h, _ = workloads.activations(cfg)
    ref, _ = oracle.ffn_decode(x_h, wg_h, wu_h, wd_h)
    wg, wu, wd, x = to_dev(wg_h), to_dev(wu_h), to_dev(wd_h), to_dev(x_h)
    m, H = x.shape
    y_lib = lib().ffn_q4k_swiglu(x, wg, wu, wd).cpu().numpy()
    stream = torch.cuda.current_stream().cuda_stream
    f = _noalloc()
    for k in range(2):  # the scratch keeps the previous call's contents; the second call must not care
        y = torch.full((m, H), float("nan"), dtype=torch.float32, device=dev())
        st = f(x.data_ptr(), m, H, cfg.inter, wg.data_ptr(), wu.data_ptr(), wd.data_ptr(), y.data_ptr(), stream)
        assert st == 0
        assert lib().q4k_last_call_kernels() >= (3 if m == 1 else 4)  # one token: no separate x kernel
        torch.cuda.synchronize()
        yn = y.cpu().numpy()
        check_close(yn, ref, TIGHT_L2, TIGHT_MAX, f"call {k}")
        assert np.array_equal(yn.view(np.uint32), y_lib.view(np.uint32))
    assert lib().q4k_check_device_error() == 0


def test_noalloc_host_buffers():
    """x and y may be mapped page-locked host memory, as for the other FFN entry points;
    pageable host memory is refused before anything is launched."""
    cfg = workloads.CONFIGS[0]
    wg_h, wu_h, wd_h = workloads.weights(cfg)
    x_h, _ = workloads.activations(cfg)
    wg, wu, wd = to_dev(wg_h), to_dev(wu_h), to_dev(wd_h)
    m, H = x_h.shape
    f = _noalloc()
    xp = torch.from_numpy(x_h).pin_memory()
    yp = torch.full((m, H), float("nan"), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream().cuda_stream
    assert f(xp.data_ptr(), m, H, cfg.inter, wg.data_ptr(), wu.data_ptr(), wd.data_ptr(), yp.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    ref, _ = oracle.ffn_decode(x_h, wg_h, wu_h, wd_h)
    check_close(yp.numpy(), ref, TIGHT_L2, TIGHT_MAX, "pinned host x, y")
    xs = np.ascontiguousarray(x_h)               # pageable numpy memory
    ys = np.zeros((m, H), np.float32)
    st = f(xs.ctypes.data, m, H, cfg.inter, wg.data_ptr(), wu.data_ptr(), wd.data_ptr(), ys.ctypes.data, stream)
    assert st == 10                              # Q4K_ERR_MEMORY
    assert lib().q4k_get_last_error() == 10
    assert not ys.any()


def test_noalloc_rejects_what_it_cannot_hold():
    f = _noalloc()
    A = torch.zeros(64, dtype=torch.float32, device=dev())  # aligned pointer; nothing is launched
    p = A.data_ptr()
    assert f(p, 9, 4096, 11008, p, p, p, p, None) == 2          # prefill shapes: Q4K_ERR_SHAPE
    assert lib().q4k_get_last_error() == 2
    assert f(p, 1, 4096, 16640, p, p, p, p, None) == 2          # beyond the 16384 dimension limit
    assert f(p, 1, 300, 4096, p, p, p, p, None) == 2             # not a multiple of 256
    assert f(None, 1, 4096, 11008, p, p, p, p, None) == 1        # Q4K_ERR_NULL
    assert lib().q4k_get_last_error() == 1
