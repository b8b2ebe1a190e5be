import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_addoption(parser):
    parser.addoption("--quick", action="store_true", default=False,
                     help="GPU parity: a stratified subset of the 216 sweep cases and no maximum-size rows")


@pytest.fixture(scope="session")
def quick(request):
    return request.config.getoption("--quick")
