import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when no GPU is present: selecting them
    # with -m gpu on a machine without one is an error of the caller.
    pass


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()
