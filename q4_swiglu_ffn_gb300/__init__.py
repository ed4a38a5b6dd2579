"""Python binding of libq4kffn.so, the sm_103a Q4_K SwiGLU feed-forward library.

Argument marshalling only: every computation runs in the library's CUDA
kernels. Tensors are torch CUDA tensors (PyTorch supplies device memory and
streams); the functions take the same names and argument order as the C ABI
in include/q4kffn.h. Importing this module raises if the library has not
been built (``python q4_swiglu_ffn_gb300/build.py``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libq4kffn.so")

Q4K_F32, Q4K_BF16 = 0, 1
STATUS = {0: "Q4K_OK", 1: "Q4K_ERR_NULL", 2: "Q4K_ERR_SHAPE", 3: "Q4K_ERR_ALIGN", 4: "Q4K_ERR_DTYPE",
          5: "Q4K_ERR_CUDA", 6: "Q4K_ERR_ARCH", 7: "Q4K_ERR_TIMEOUT", 8: "Q4K_ERR_NOMEM", 9: "Q4K_ERR_RANGE",
          10: "Q4K_ERR_MEMORY"}

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python q4_swiglu_ffn_gb300/build.py`")

lib = ctypes.CDLL(LIB_PATH)
PREFILL_READY = True

_i64, _sz, _p, _int = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
_SIGS = {
    "q4k_weight_bytes": (_sz, [_i64, _i64]),
    "q8_1_bytes": (_sz, [_i64, _i64]),
    "q4k_quantize_weights": (_int, [_p, _int, _i64, _i64, _p, _p]),
    "q8_1_quantize_act": (_int, [_p, _int, _i64, _i64, _p, _p]),
    "ffn_q4k_swiglu": (_int, [_p, _i64, _i64, _i64, _p, _p, _p, _p, _p]),
    "ffn_q4k_swiglu_ex": (_int, [_p, _int, _i64, _i64, _i64, _p, _p, _p, _p, _p, _sz, _p]),
    "ffn_q4k_swiglu_q8_1": (_int, [_p, _int, _i64, _i64, _i64, _p, _p, _p, _p, _p, _sz, _p]),
    "ffn_q4k_swiglu_ex_y": (_int, [_p, _int, _i64, _i64, _i64, _p, _p, _p, _p, _int, _p, _sz, _p]),
    "ffn_q4k_q8_1_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "ffn_q4k_q8_1_workspace_h_offset": (_sz, [_i64, _i64, _i64]),
    "ffn_q4k_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "ffn_q4k_workspace_h_q8_1_offset": (_sz, [_i64, _i64, _i64]),
    "q4k_dequantize": (_int, [_p, _i64, _i64, _p, _p]),
    "q6k_weight_bytes": (_sz, [_i64, _i64]),
    "q6k_gemv_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "q6k_gemv": (_int, [_p, _int, _i64, _i64, _i64, _p, _p, _p, _sz, _p]),
    "q6k_dequantize": (_int, [_p, _i64, _i64, _p, _p]),
    "q4k_check_device_error": (_int, [_p]),
    "q4k_test_bounded_wait": (_int, [ctypes.c_uint64, _p]),
    "q4k_set_profile_events": (_int, [_p, _int]),
    "q4k_get_last_error": (_int, []),
    "q4k_last_call_kernels": (_int, []),
    "q4k_status_string": (ctypes.c_char_p, [_int]),
    "q4k_bench_int8_mma": (_int, [_i64, ctypes.POINTER(ctypes.c_double), _p]),
    "q4k_bench_tcgen05_issue": (_int, [_int, _int, _i64, ctypes.POINTER(ctypes.c_double), _p]),
    "q4k_mmq_fp8": (_int, [_p, _i64, _i64, _p, _i64, _p, _p, _sz, _p]),
    "q4k_mmq_fp8_workspace_bytes": (_sz, [_i64, _i64]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class Q4KError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({lib.q4k_status_string(status).decode()})")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise Q4KError(status, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


_current_raw_stream = None  # () -> the current device's current CUDA stream, as a raw handle


def _stream(stream):
    """The stream argument as a raw handle; None is PyTorch's current stream."""
    global _current_raw_stream
    if stream is None:
        if _current_raw_stream is None:
            import torch
            get_raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            get_dev = getattr(torch._C, "_cuda_getDevice", None)
            if get_raw is not None and get_dev is not None:
                torch.cuda.init()
                _current_raw_stream = lambda: get_raw(get_dev())
            else:  # same handle through the public API (slower: builds a Stream object)
                _current_raw_stream = lambda: torch.cuda.current_stream().cuda_stream
        return _current_raw_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


_DTYPES = None  # {torch.float32: Q4K_F32, torch.bfloat16: Q4K_BF16}


def _dtype_code(t) -> int:
    global _DTYPES
    if _DTYPES is None:
        import torch
        _DTYPES = {torch.float32: Q4K_F32, torch.bfloat16: Q4K_BF16}
    code = _DTYPES.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported activation dtype {t.dtype}")
    return code


def q4k_weight_bytes(rows: int, cols: int) -> int:
    return lib.q4k_weight_bytes(rows, cols)


def q8_1_bytes(m: int, k: int) -> int:
    return lib.q8_1_bytes(m, k)


def ffn_q4k_workspace_bytes(m: int, hidden: int, inter: int) -> int:
    return lib.ffn_q4k_workspace_bytes(m, hidden, inter)


def ffn_q4k_q8_1_workspace_bytes(m: int, hidden: int, inter: int) -> int:
    return lib.ffn_q4k_q8_1_workspace_bytes(m, hidden, inter)


def ffn_q4k_q8_1_workspace_h_offset(m: int, hidden: int, inter: int) -> int:
    return lib.ffn_q4k_q8_1_workspace_h_offset(m, hidden, inter)


def ffn_q4k_workspace_h_q8_1_offset(m: int, hidden: int, inter: int) -> int:
    return lib.ffn_q4k_workspace_h_q8_1_offset(m, hidden, inter)


def q4k_quantize_weights(W, out=None, stream=None):
    """W: [rows, cols] float32/bf16 CUDA tensor -> uint8 Q4_K blocks [rows, cols/256, 144]."""
    import torch
    rows, cols = W.shape
    if out is None:
        out = torch.empty((rows, cols // 256, 144), dtype=torch.uint8, device=W.device)
    _check(lib.q4k_quantize_weights(_ptr(W), _dtype_code(W), rows, cols, _ptr(out), _stream(stream)),
           "q4k_quantize_weights")
    return out


def q8_1_quantize_act(x, out=None, stream=None):
    """x: [m, k] float32/bf16 CUDA tensor -> planar Q8_1 bytes (uint8, q8_1_bytes(m, k))."""
    import torch
    m, k = x.shape
    if out is None:
        out = torch.empty(q8_1_bytes(m, k), dtype=torch.uint8, device=x.device)
    _check(lib.q8_1_quantize_act(_ptr(x), _dtype_code(x), m, k, _ptr(out), _stream(stream)), "q8_1_quantize_act")
    return out


def ffn_q4k_swiglu(x, W_gate, W_up, W_down, y=None, stream=None):
    """y = W_down (silu(W_gate x) * (W_up x)); x float32 [m, hidden] -> y float32 [m, hidden]."""
    m, hidden = x.shape
    inter = W_gate.shape[0]
    if y is None:
        import torch
        y = torch.empty((m, hidden), dtype=torch.float32, device=x.device)
    _check(lib.ffn_q4k_swiglu(_ptr(x), m, hidden, inter, _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(y),
                              _stream(stream)), "ffn_q4k_swiglu")
    return y


def ffn_q4k_swiglu_ex(x, W_gate, W_up, W_down, workspace, y=None, stream=None):
    """As ffn_q4k_swiglu with float32 or bf16 x and a caller workspace (uint8 CUDA tensor; any contents)."""
    import torch
    m, hidden = x.shape
    inter = W_gate.shape[0]
    if y is None:
        y = torch.empty((m, hidden), dtype=torch.float32, device=x.device)
    _check(lib.ffn_q4k_swiglu_ex(_ptr(x), _dtype_code(x), m, hidden, inter, _ptr(W_gate), _ptr(W_up),
                                 _ptr(W_down), _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)),
           "ffn_q4k_swiglu_ex")
    return y


def ffn_q4k_swiglu_ex_y(x, W_gate, W_up, W_down, workspace, y):
    """As ffn_q4k_swiglu_ex, writing y as float32 or bf16 (the dtype of the given y tensor)."""
    m, hidden = x.shape
    inter = W_gate.shape[0]
    _check(lib.ffn_q4k_swiglu_ex_y(_ptr(x), _dtype_code(x), m, hidden, inter, _ptr(W_gate), _ptr(W_up),
                                   _ptr(W_down), _ptr(y), _dtype_code(y), _ptr(workspace), workspace.numel(),
                                   _stream(None)), "ffn_q4k_swiglu_ex_y")
    return y


def ffn_q4k_swiglu_q8_1(x, W_gate, W_up, W_down, workspace, y=None, stream=None):
    """The FFN with Q8_1 activations at every m (x float32 or bf16; caller workspace, uint8 CUDA tensor)."""
    import torch
    m, hidden = x.shape
    inter = W_gate.shape[0]
    if y is None:
        y = torch.empty((m, hidden), dtype=torch.float32, device=x.device)
    _check(lib.ffn_q4k_swiglu_q8_1(_ptr(x), _dtype_code(x), m, hidden, inter, _ptr(W_gate), _ptr(W_up),
                                   _ptr(W_down), _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)),
           "ffn_q4k_swiglu_q8_1")
    return y


def q4k_dequantize(q, rows: int, cols: int, out=None, stream=None):
    """Test hook: Q4_K blocks -> float32 [rows, cols]."""
    import torch
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=q.device)
    _check(lib.q4k_dequantize(_ptr(q), rows, cols, _ptr(out), _stream(stream)), "q4k_dequantize")
    return out


def q6k_weight_bytes(rows: int, cols: int) -> int:
    return lib.q6k_weight_bytes(rows, cols)


def q6k_gemv_workspace_bytes(m: int, n: int, k: int) -> int:
    return lib.q6k_gemv_workspace_bytes(m, n, k)


def q6k_gemv(x, W, workspace, y=None, stream=None):
    """y [m, n] = x [m, k] . W^T for Q6_K blocks W (uint8 [n, k/256, 210]); x float32 or bf16."""
    import torch
    m, k = x.shape
    n = W.shape[0]
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    _check(lib.q6k_gemv(_ptr(x), _dtype_code(x), m, n, k, _ptr(W), _ptr(y), _ptr(workspace), workspace.numel(),
                        _stream(stream)), "q6k_gemv")
    return y


def q6k_dequantize(q, rows: int, cols: int, out=None, stream=None):
    """Test hook: Q6_K blocks -> float32 [rows, cols]."""
    import torch
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=q.device)
    _check(lib.q6k_dequantize(_ptr(q), rows, cols, _ptr(out), _stream(stream)), "q6k_dequantize")
    return out


def q4k_check_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status code."""
    return lib.q4k_check_device_error(_stream(stream))


def q4k_test_bounded_wait(limit_ns: int, stream=None) -> None:
    """Enqueue a wait that nothing completes; it gives up after limit_ns and records a timeout."""
    _check(lib.q4k_test_bounded_wait(int(limit_ns), _stream(stream)), "q4k_test_bounded_wait")


def q4k_set_profile_events(events) -> None:
    """Record torch.cuda.Event pairs around each kernel of the following FFN calls (None: off)."""
    global _prof_keep
    if not events:
        _check(lib.q4k_set_profile_events(None, 0), "q4k_set_profile_events")
        _prof_keep = None
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _prof_keep = arr  # the library keeps the pointer; keep the array alive
    _check(lib.q4k_set_profile_events(arr, len(events)), "q4k_set_profile_events")


_prof_keep = None


def q4k_last_call_kernels() -> int:
    """Kernels the last FFN or Q6_K GEMV call on this thread launched (benchmark hook)."""
    return lib.q4k_last_call_kernels()


def q4k_mmq_fp8_workspace_bytes(m: int, k: int) -> int:
    return lib.q4k_mmq_fp8_workspace_bytes(m, k)


def q4k_mmq_fp8(xq8, m, k, W, workspace=None, out=None, stream=None):
    """Q4_K x Q8_1 GEMM on the FP8 tensor path: xq8 planar Q8_1 bytes of [m, k] activations,
    W Q4_K bytes [n, k/256, 144] -> out float32 [m, n] (out[t][r] = sum_k W[r][k] x[t][k])."""
    import torch
    n = W.shape[0]
    if workspace is None:
        workspace = torch.empty(q4k_mmq_fp8_workspace_bytes(m, k), dtype=torch.uint8, device=W.device)
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=W.device)
    _check(lib.q4k_mmq_fp8(_ptr(xq8), m, k, _ptr(W), n, _ptr(out), _ptr(workspace), workspace.numel(),
                           _stream(stream)), "q4k_mmq_fp8")
    return out


def q4k_bench_int8_mma(iters: int, stream=None) -> float:
    """Enqueues the int8 tensor-rate kernel; returns the integer operations of the launch (benchmark hook)."""
    ops = ctypes.c_double(0.0)
    _check(lib.q4k_bench_int8_mma(iters, ctypes.byref(ops), _stream(stream)), "q4k_bench_int8_mma")
    return ops.value


def q4k_bench_tcgen05_issue(n: int, issuers: int, iters: int, stream=None) -> float:
    """SM cycles per tcgen05.mma (M 128, N n, K 16) of one of `issuers` issuing threads per CTA
    (benchmark hook; runs on the stream and waits for it)."""
    cyc = ctypes.c_double(0.0)
    _check(lib.q4k_bench_tcgen05_issue(n, issuers, iters, ctypes.byref(cyc), _stream(stream)),
           "q4k_bench_tcgen05_issue")
    return cyc.value


def q4k_get_last_error() -> int:
    return lib.q4k_get_last_error()
