import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running exhaustive check (opt-in via KVFP8_SLOW=1)")


def pytest_collection_modifyitems(config, items):
    if os.environ.get("KVFP8_SLOW") == "1":
        return
    skip = pytest.mark.skip(reason="exhaustive check; set KVFP8_SLOW=1 to run")
    for item in items:
        if "slow" in item.keywords:
            item.add_marker(skip)
