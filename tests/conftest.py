import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def load_golden(name):
    import json
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def tg():
    """The Python binding, with libtilegemm built in-tree first (nvcc, sm_103a)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_tg_build", os.path.join(ROOT, "tiled_gemm_layouts_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import tiled_gemm_layouts_gb300 as tgmod
    return tgmod
