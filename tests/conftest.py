import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running GPU parity case")


def pytest_addoption(parser):
    parser.addoption("--full-sweep", action="store_true", default=False,
                     help="run all 216 sweep cases instead of the default stratified subset")
    parser.addoption("--max-size", action="store_true", default=False,
                     help="run the parity cases at the ABI's maximum sizes (2M-token rows; minutes of oracle time)")


@pytest.fixture(scope="session")
def full_sweep(request):
    return request.config.getoption("--full-sweep")


@pytest.fixture(scope="session")
def max_size(request):
    return request.config.getoption("--max-size")
