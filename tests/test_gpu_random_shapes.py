"""Seeded random shapes across the dispatch branches: decode passes (m <= 24), the unsplit and
split down GEMV, the prefill GEMM with and without K slices, both activation paths."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import (ACCEPT_L2, ACCEPT_MAX, TIGHT_L2, TIGHT_MAX, check_close, dev, guarded_f32, guards_intact,
                            lib, to_dev, torch)

pytestmark = pytest.mark.gpu

_rng = np.random.default_rng(2026)
CASES = [(int(256 * _rng.integers(1, 17)), int(256 * _rng.integers(1, 17)), int(m))
         for m in (1, 2, 3, 5, 7, 8, 11, 19, 24, 25, 40, 130)]


@pytest.mark.parametrize("H,I,m", CASES)
def test_random_shape_both_paths(H, I, m):
    c = workloads.small_config(H, I, m, "f32", ("channels", 0.01, 30.0))
    wg, wu, wd = workloads.weights(c)
    dg, du, dd = to_dev(wg), to_dev(wu), to_dev(wd)
    x, _ = workloads.activations(c)
    xd = to_dev(x)
    # float32 entry: decode numerics up to 24 tokens, Q8_1 prefill above
    buf, y = guarded_f32(m * H)
    ws = torch.empty(lib().ffn_q4k_workspace_bytes(m, H, I), dtype=torch.uint8, device=dev())
    lib().ffn_q4k_swiglu_ex(xd, dg, du, dd, ws, y=y.view(m, H))
    torch.cuda.synchronize()
    assert guards_intact(buf)
    y32 = y.view(m, H).cpu().numpy()
    if m <= 24:
        ref, _ = oracle.ffn_decode(x, wg, wu, wd)
        check_close(y32, ref, TIGHT_L2, TIGHT_MAX, "float32 entry (decode)")
    else:
        check_close(y32, oracle.ffn_prefill(x, wg, wu, wd)["y"], ACCEPT_L2, ACCEPT_MAX, "float32 entry (prefill)")
    # Q8_1 entry: the Q8_1 oracle at every m
    buf8, y8 = guarded_f32(m * H)
    ws8 = torch.empty(lib().ffn_q4k_q8_1_workspace_bytes(m, H, I), dtype=torch.uint8, device=dev())
    lib().ffn_q4k_swiglu_q8_1(xd, dg, du, dd, ws8, y=y8.view(m, H))
    torch.cuda.synchronize()
    assert guards_intact(buf8)
    check_close(y8.view(m, H).cpu().numpy(), oracle.ffn_prefill(x, wg, wu, wd)["y"], ACCEPT_L2, ACCEPT_MAX,
                "Q8_1 entry")
    assert lib().q4k_check_device_error() == 0
