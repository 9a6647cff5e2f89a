import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); calls the C ABI")


@pytest.fixture(scope="session")
def sdpa_lib():
    """The built C-ABI library (built in-tree on first use)."""
    from scaled_dot_product_fwd_gb300 import build as b
    b.build()
    import scaled_dot_product_fwd_gb300 as s
    return s.load_library()


@pytest.fixture(scope="session")
def cuda():
    """torch with a CUDA device; a GPU test without one fails instead of skipping."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for a gpu-marked test")
    from scaled_dot_product_fwd_gb300 import build as b
    b.build()
    return torch
