"""The allocation-free decode entry point agrees with ffn_q4k_swiglu.

ffn_q4k_swiglu_noalloc serves callers that cannot call cudaMalloc (a server
whose pool owns all device memory, a loop that cannot take cudaMalloc's
device-wide synchronisation): it runs the decode kernels on a static scratch
array inside the library. This file is collected last so that a run stopping
at the first failure has already run every other test; it also passes alone.
"""
import ctypes

import numpy as np
import pytest

import workloads
from tests.gpu_util import dev, lib, rel_l2, to_dev, torch

pytestmark = pytest.mark.gpu

TOL = 2e-5  # the decode tolerance used by the other decode tests


def _noalloc():
    f = lib().lib.ffn_q4k_swiglu_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + [ctypes.c_void_p] * 5
    return f


@pytest.mark.parametrize("cfg_index", [1, 2])
def test_noalloc_matches_ffn_q4k_swiglu_twice(cfg_index):
    cfg = workloads.CONFIGS[cfg_index]
    wg, wu, wd = [to_dev(a) for a in workloads.weights(cfg)]
    x = to_dev(workloads.activations(cfg)[0])
    m, H = x.shape
    y_ref = lib().ffn_q4k_swiglu(x, wg, wu, wd)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    f = _noalloc()
    for _ in range(2):  # the scratch keeps the previous call's contents; the second call must not care
        y = torch.full((m, H), float("nan"), dtype=torch.float32, device=dev())
        st = f(x.data_ptr(), m, H, cfg.inter, wg.data_ptr(), wu.data_ptr(), wd.data_ptr(), y.data_ptr(), stream)
        assert st == 0
        torch.cuda.synchronize()
        assert rel_l2(y.cpu().numpy(), y_ref.cpu().numpy()) <= TOL


def test_noalloc_rejects_what_it_cannot_hold():
    f = _noalloc()
    A = torch.zeros(64, dtype=torch.float32, device=dev())  # aligned pointer; nothing is launched
    p = A.data_ptr()
    assert f(p, 9, 4096, 11008, p, p, p, p, None) == 2          # prefill shapes: Q4K_ERR_SHAPE
    assert f(p, 1, 4096, 16640, p, p, p, p, None) == 2          # beyond the 16384 dimension limit
    assert f(p, 1, 300, 4096, p, p, p, p, None) == 2             # not a multiple of 256
    assert f(None, 1, 4096, 11008, p, p, p, p, None) == 1        # Q4K_ERR_NULL
