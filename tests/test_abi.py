"""The C-ABI library builds, loads and exports every symbol include/q4kffn.h declares;
host-side argument checks run without a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "q4kffn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z][a-z0-9_]*)\s*\(", text)
    skip = {"if", "while", "for", "sizeof", "return", "defined"}
    return sorted({n for n in names if n not in skip})


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "ffn_q4k_swiglu" in names and "q8_1_quantize_act" in names and "q4k_quantize_weights" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_byte_size_helpers(lib):
    lib.q4k_weight_bytes.restype = ctypes.c_size_t
    lib.q4k_weight_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    lib.q8_1_bytes.restype = ctypes.c_size_t
    lib.q8_1_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    assert lib.q4k_weight_bytes(11008, 4096) == 11008 * 16 * 144
    assert lib.q4k_weight_bytes(4096, 11008) == 4096 * 43 * 144
    assert lib.q4k_weight_bytes(10, 300) == 0 and lib.q4k_weight_bytes(0, 256) == 0
    assert lib.q8_1_bytes(512, 4096) == 512 * 4096 + 512 * 128 * 8
    assert lib.q8_1_bytes(0, 256) == 0


def _ffn(lib, x, m, h, i, wg, wu, wd, y):
    f = lib.ffn_q4k_swiglu
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + [ctypes.c_void_p] * 5
    return f(x, m, h, i, wg, wu, wd, y, None)


def test_argument_errors_before_any_launch(lib):
    A = 1 << 20  # a 16-byte aligned fake address; never dereferenced because validation fails first
    assert _ffn(lib, None, 1, 256, 768, A, A, A, A) == 1            # Q4K_ERR_NULL
    assert _ffn(lib, A, 1, 256, 768, A, None, A, A) == 1
    assert _ffn(lib, A, 0, 256, 768, A, A, A, A) == 2               # m = 0
    assert _ffn(lib, A, 1, 300, 768, A, A, A, A) == 2               # hidden % 256 != 0
    assert _ffn(lib, A, 1, 256, 700, A, A, A, A) == 2               # inter % 256 != 0
    assert _ffn(lib, A, 1, 1 << 21, 256, A, A, A, A) == 2           # beyond the size limit
    assert _ffn(lib, A + 4, 1, 256, 768, A, A, A, A) == 3           # misaligned x
    assert _ffn(lib, A, 1, 256, 768, A, A, A + 8, A) == 3           # misaligned W_down
    lib.q4k_get_last_error.restype = ctypes.c_int
    assert lib.q4k_get_last_error() == 3
    q = lib.q8_1_quantize_act
    q.restype = ctypes.c_int
    q.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    assert q(A, 7, 1, 256, A, None) == 4                             # Q4K_ERR_DTYPE
    assert q(A, 0, 1, 100, A, None) == 2
    w = lib.q4k_quantize_weights
    w.restype = ctypes.c_int
    w.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    assert w(None, 0, 4, 256, A, None) == 1
    assert w(A, 0, 4, 255, A, None) == 2
    b = lib.q4k_bench_tcgen05_issue
    b.restype = ctypes.c_int
    b.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p]
    c = ctypes.c_double(0.0)
    assert b(128, 1, 64, None, None) == 1                            # no result pointer
    assert b(100, 1, 64, ctypes.byref(c), None) == 2                 # N not 64, 128 or 256
    assert b(256, 2, 64, ctypes.byref(c), None) == 2                 # 512 accumulator columns
    assert b(128, 3, 64, ctypes.byref(c), None) == 2                 # issuers not 1, 2 or 4
    assert b(128, 1, 0, ctypes.byref(c), None) == 2                  # no rounds


def test_status_strings(lib):
    lib.q4k_status_string.restype = ctypes.c_char_p
    for s in range(11):
        assert lib.q4k_status_string(s)
    assert b"unknown" in lib.q4k_status_string(99)
