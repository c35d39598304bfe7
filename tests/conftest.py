import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_sessionstart(session):
    """Build libkvq (skipped when up to date) and the oracle before any test
    imports them."""
    spec = importlib.util.spec_from_file_location(
        "kvq_build", os.path.join(ROOT, "quantized_paged_kv_quantize_gb300", "_build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import oracle
    oracle.build()


@pytest.fixture(autouse=True)
def _canaries():
    """After every test, the canary bands around the device buffers it handed
    to the kernels (tests/_helpers.guarded) must be intact."""
    yield
    if "_helpers" in sys.modules:
        sys.modules["_helpers"].check_guards()
