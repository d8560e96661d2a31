import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU-side oracle work")


_CACHE = {}


def cached_workload(name, *args, **kw):
    """Workloads are deterministic; build each one once per test session."""
    import workloads

    key = (name, args, tuple(sorted(kw.items())))
    if key not in _CACHE:
        fn = workloads.NAMED.get(name) or getattr(workloads, name)
        _CACHE[key] = fn(*args, **kw)
    return _CACHE[key]


@pytest.fixture(scope="session")
def wl_cache():
    return cached_workload
