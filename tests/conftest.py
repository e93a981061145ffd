import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


@pytest.fixture(autouse=True)
def _guards_intact():
    """After every test: the guard regions around the outputs the GPU helpers
    allocated (tests/gpu_cases.py) still hold their patterns."""
    yield
    mod = sys.modules.get("tests.gpu_cases")
    if mod is not None and mod._live:
        mod.assert_guards_intact()
