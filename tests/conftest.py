import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def mnb():
    """The CUDA library's Python binding (built in-tree on first use)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_weight_matmulnbits_gb300 as m
    m.load()
    return m


@pytest.fixture(scope="session")
def G(mnb):
    """GPU-test helpers (tests/_gpu.py), loaded once the library is."""
    from tests import _gpu
    return _gpu
