import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (runs the CUDA library)")
    config.addinivalue_line(
        "markers", "slow: statistical or full-size case (still in the suite)")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library, built in-tree if needed (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_drafter_verify_gb300 as dv
    return dv
