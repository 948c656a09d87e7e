import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def load_golden(name):
    import json
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture
def golden():
    return load_golden


@pytest.fixture(scope="session")
def native_lib():
    """Builds (if stale) and loads libpagedkv.so; no CUDA call is made."""
    from paged_kv_cache_138_gb300 import build
    build.build()
    from paged_kv_cache_138_gb300 import _lib
    return _lib.lib()


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False
