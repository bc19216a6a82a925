import os
import sys

import pytest

_TESTS = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_TESTS)
for p in (_ROOT, _TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs on a GB300)")
    config.addinivalue_line("markers", "slow: full-size workloads")


def load_build_module():
    """deterministic_fixed_order_gb300/build.py, loaded by path (the package
    import itself requires the built library)."""
    import importlib.util
    path = os.path.join(_ROOT, "deterministic_fixed_order_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_detfold_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


# Build the CUDA library (if stale) before any test module imports the package.
load_build_module().build()
