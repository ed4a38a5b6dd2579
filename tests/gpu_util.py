"""Helpers shared by the GPU tests: device tensors from numpy, error metrics, guard bands."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

GUARD = 4096  # floats of guard band on each side of an output


def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def lib():
    import q4_swiglu_ffn_gb300 as q
    return q


def to_dev(a: np.ndarray):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:   # bf16 bit patterns
        return torch.from_numpy(a.view(np.int16)).to(dev()).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev())


def guarded_f32(n: int):
    """A float32 buffer of n elements with NaN-pattern guard bands on both sides."""
    buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=torch.float32, device=dev())
    return buf, buf[GUARD:GUARD + n]


def guards_intact(buf) -> bool:
    g = torch.cat([buf[:GUARD], buf[-GUARD:]])
    return bool(torch.isnan(g).all().item())


def rel_l2(y, ref) -> float:
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


def rel_max(y, ref) -> float:
    """Element-wise error: max |y - ref| over max |ref| (both over the whole output)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(y - ref)) / max(np.max(np.abs(ref)), 1e-300))


# Tolerances. Acceptance for the FFN output: L2-relative error <= 1e-3, and
# every element within 1e-3 of the output's largest magnitude. Paths whose
# arithmetic sits far below that (float32 activations carried as fp16 hi + lo,
# about 22 bits, exact weights, float32 sums) also meet TIGHT_L2 / TIGHT_MAX,
# which a dropped term or a wrong index could not.
ACCEPT_L2, ACCEPT_MAX = 1e-3, 1e-3
TIGHT_L2, TIGHT_MAX = 2e-5, 1e-4

_REPORT = []  # (test id, what, rel_l2, rel_max), printed by the session summary


def check_close(y, ref, l2, elem, what="y"):
    """Asserts rel_l2(y, ref) <= l2 and rel_max(y, ref) <= elem, and records both."""
    import os
    e2, em = rel_l2(y, ref), rel_max(y, ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    _REPORT.append((test, what, e2, em))
    assert e2 <= l2 and em <= elem, f"{what}: rel_l2 {e2:.3g} (bound {l2:g}), rel_max {em:.3g} (bound {elem:g})"
    return e2, em


def report_lines():
    return [f"{t}  {w}: rel_l2 {a:.3e}  rel_max {b:.3e}" for (t, w, a, b) in _REPORT]
