import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libneo")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def gpu_lib():
    """Builds (if stale) and loads libneo; a GPU test fails loudly without either."""
    import torch

    from attention_neo_qknorm_gb300 import neo
    from attention_neo_qknorm_gb300.build import build

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    return neo.load_library()
