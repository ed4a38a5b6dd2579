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
