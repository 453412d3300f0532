import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libscute.so")


@pytest.fixture(scope="session")
def gpu_lib():
    """The loaded CUDA library; GPU tests fail loudly when it is missing."""
    import lora_normal_form_gb300 as scute
    scute.load()
    return scute
