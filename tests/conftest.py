import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")


def pytest_sessionstart(session):
    """GPU runs build the library first (the build is incremental and takes seconds)."""
    markexpr = session.config.getoption("markexpr", "") or ""
    if "gpu" in markexpr and "not gpu" not in markexpr:
        import __graft_entry__
        __graft_entry__._build_module().build()


def pytest_terminal_summary(terminalreporter):
    """Prints, for every parity check the GPU tests made, the L2-relative and element-wise errors."""
    mod = sys.modules.get("tests.gpu_util")
    lines = mod.report_lines() if mod is not None else []
    if lines:
        terminalreporter.section("parity errors (rel_l2 = |y-ref|_2/|ref|_2, rel_max = max|y-ref|/max|ref|)")
        for line in lines:
            terminalreporter.write_line(line)
