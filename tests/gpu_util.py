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
