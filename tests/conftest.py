import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def golden():
    from tests._golden import load
    return load


@pytest.fixture(scope="session", autouse=True)
def _kvq_library_under_test(request):
    """With KVQ_TEST_DEBUG=1 in the environment, every test that goes through
    the binding runs on the debug build (libkvq_debug.so: each global access
    checked against its array's extent, KVQ_FLAG_OOB on a miss), so the
    whole GPU suite doubles as an out-of-bounds sweep: any check that fires
    shows up as a nonzero status word in the test that caused it."""
    if os.environ.get("KVQ_TEST_DEBUG") != "1":
        yield
        return
    from quantized_kv_decode_gb300 import _lib, build
    handle = _lib.load(build.build(debug=True))
    assert handle.kvq_debug_checks() == 1
    prev = _lib.use(handle)
    try:
        yield
    finally:
        _lib.use(prev)
