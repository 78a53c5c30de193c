import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libep.so")
    config.addinivalue_line("markers", "slow: large CPU oracle runs")


def pytest_collection_modifyitems(config, items):
    """A GPU test that stalls (a kernel that never returns) ends its test process after ten
    minutes, with every thread's stack printed, instead of holding the GPU until an outer limit
    (needs the pytest-timeout plugin; without it nothing changes)."""
    if not config.pluginmanager.hasplugin("timeout"):
        return
    for item in items:
        if item.get_closest_marker("gpu") and not item.get_closest_marker("timeout"):
            item.add_marker(pytest.mark.timeout(600, method="thread"))
