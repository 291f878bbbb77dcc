import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "full_size: runs the benchmark's full-size workload "
                            "(collected last, so that a run stopping at its first failure has "
                            "run every smaller test first)")


def pytest_collection_modifyitems(config, items):
    items.sort(key=lambda item: item.get_closest_marker("full_size") is not None)


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
