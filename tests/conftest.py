import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _build_libraries():
    """Build the CUDA library (nvcc cross-compiles without a GPU) and the oracle."""
    path = os.path.join(ROOT, "fp8_paged_kv_reshape_gb300", "_build.py")
    spec = importlib.util.spec_from_file_location("_kvfp8_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import oracle.build

    oracle.build.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running exhaustive check (opt-in via KVFP8_SLOW=1)")
    _build_libraries()


def pytest_collection_modifyitems(config, items):
    if os.environ.get("KVFP8_SLOW") == "1":
        return
    skip = pytest.mark.skip(reason="exhaustive check; set KVFP8_SLOW=1 to run")
    for item in items:
        if "slow" in item.keywords:
            item.add_marker(skip)
