import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU-side oracle work")


@pytest.fixture(autouse=True)
def _release_device_temporaries():
    yield
    mod = sys.modules.get("gpu_util")
    if mod is not None:
        mod.release()
