import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # GPU tests need a device; on a machine without one they are skipped only
    # when not explicitly selected with -m gpu (then they fail loudly).
    pass
