import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (seconds to minutes)")


def pytest_collection_modifyitems(config, items):
    # GPU tests on a machine without a GPU are an error of selection, not a skip:
    # the CPU suite is selected with -m "not gpu".
    pass


@pytest.fixture(scope="session")
def oracle():
    from oracle import h3q_oracle
    return h3q_oracle


@pytest.fixture(scope="session")
def lib():
    """The CUDA library through its Python binding (loads libh3q.so, builds it if absent)."""
    import w8a8_int8_linear_h3q_gb300 as h3q
    h3q.load()
    return h3q
