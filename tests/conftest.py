import importlib.util
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _build_cuda_library():
    """Compile libss.so in-tree if it is missing or stale (nvcc cross-compiles
    without a GPU). Loaded by file path so that the package (which refuses to
    import without the library) is not imported first."""
    if not (os.environ.get("NVCC") or shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        return
    path = os.path.join(ROOT, "sampled_softmax_output_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_ss_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    _build_cuda_library()


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
