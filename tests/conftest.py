import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running on CPU")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without a GPU fails loudly rather than skipping:
    # the driver selects them with -m gpu only where a GPU exists.
    pass
