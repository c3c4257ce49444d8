import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes of host work)")


def pytest_collection_modifyitems(config, items):
    # Keep collection order stable: files sorted by name, so the file named
    # test_zz_* runs last.
    items.sort(key=lambda it: (os.path.basename(str(it.fspath)), 0))


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
