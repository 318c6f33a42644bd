import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled libmha.so")


def pytest_collection_modifyitems(config, items):
    # A gpu-marked test on a machine without CUDA is a hard error, not a skip:
    # the driver only selects them with -m gpu on a GPU machine.
    pass


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle
