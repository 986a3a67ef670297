import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkvc")
    config.addinivalue_line("markers", "slow: full-size case, minutes of CPU work")


@pytest.fixture(scope="session")
def cuda_layer_module():
    """The product binding, or a skip when no GPU is present (CPU runs)."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rank_quantized_kv_gb300 as kvc

    return kvc
