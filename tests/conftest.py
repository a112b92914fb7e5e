import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libfs.so")
    config.addinivalue_line("markers", "slow: long-running oracle comparison at full workload size")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def fs():
    """The CUDA library binding; fails loudly (never skips) when it cannot load."""
    from mixture_experts_layer_expert_gb300 import fs as _fs
    _fs.lib()
    return _fs


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
