import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case")


def pytest_collection_modifyitems(config, items):
    # tests whose name says they run on the GPU must carry the marker
    for it in items:
        if "gpu" in it.nodeid.split("::")[0] and "gpu" not in it.keywords:
            it.add_marker(pytest.mark.gpu)
