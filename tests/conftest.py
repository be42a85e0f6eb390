import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def _stale(lib_path, src_dirs):
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    for d in src_dirs:
        for f in os.listdir(d):
            if f.endswith((".cu", ".cuh", ".cpp", ".h")) and os.path.getmtime(os.path.join(d, f)) > t:
                return True
    return False


@pytest.fixture(scope="session")
def librx():
    """The native library, (re)built in-tree when missing or older than its sources."""
    from prefix_shared_kv_gb300 import build, rx
    if _stale(build.LIB, [build.CSRC, build.INCLUDE]):
        build.build()
    return rx.lib()


@pytest.fixture(scope="session")
def cuda(librx):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
