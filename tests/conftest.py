import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA path's Python binding, with the extension built and a GPU present."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import megatron_tensor_transformer_column_gb300 as tp
    tp.load()  # raises if the extension is missing or fails to load
    return tp
