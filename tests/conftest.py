import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    """A gpu-marked test on a machine without a GPU is an error of the
    invocation, not something to skip silently: the CPU suite is run with
    ``-m "not gpu"``."""
    return None
