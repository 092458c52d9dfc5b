import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    return torch.device("cuda:0")

# The randomised oracle invariants need hypothesis, which only the CPU test
# environment provides; where it is missing the module is not collected at all
# (it holds CPU-only tests, so a GPU run loses nothing and reports no skip).
collect_ignore = []
try:
    import hypothesis  # noqa: F401
except ImportError:
    collect_ignore.append("test_oracle_properties.py")
