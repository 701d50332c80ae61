import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds of CPU")


def pytest_collection_modifyitems(config, items):
    # files named test_zz_* run after every other test file
    items.sort(key=lambda it: os.path.basename(str(it.fspath)).startswith("test_zz_"))
