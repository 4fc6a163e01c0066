import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    # Build the native library in-tree if it is missing (nvcc cross-compiles
    # here and builds natively on the GPU machine).
    import importlib.util
    path = os.path.join(ROOT, "bit_quantized_moe_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("qmv_build", path)
    qbuild = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(qbuild)
    if not os.path.exists(qbuild.LIB):
        qbuild.build()
