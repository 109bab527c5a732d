import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libqmm.so")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


def load_builder():
    """The package's build module, loaded by path (importing the package
    itself requires the built library)."""
    import importlib.util
    path = os.path.join(ROOT, "block_quantized_matmul_q4_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("qmm_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="session")
def built_lib():
    return load_builder().build()
