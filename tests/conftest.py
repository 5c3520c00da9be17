import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs through the C-ABI library)")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of oracle time)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def lct_lib():
    """The C-ABI library, built for sm_103a if it is missing (no GPU needed to load it)."""
    from lossless_bf16_tensor_gb300 import build as b
    b.build_library()
    from lossless_bf16_tensor_gb300 import binding
    return binding
