"""Host-side checks of the launch plans without a GPU: tests/host_plans.cpp calls the
library's plan functions over a grid of shapes and SM counts and checks tile and chunk
counts and workspace offsets (alignment, order, bounds)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plans_are_consistent(tmp_path):
    import __graft_entry__
    lib = __graft_entry__._build_module().build()
    cxx = shutil.which("g++")
    cuda_inc = "/usr/local/cuda/include"
    if not cxx or not os.path.isdir(cuda_inc):
        pytest.skip("needs g++ and the CUDA headers")
    exe = str(tmp_path / "host_plans")
    pkg = os.path.dirname(lib)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", os.path.join(pkg, "csrc"), "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "host_plans.cpp"), "-L", pkg, "-lq4kffn",
                    "-Wl,-rpath," + pkg, "-o", exe], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok"), r.stdout
