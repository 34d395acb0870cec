import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libsab.so")
    config.addinivalue_line("markers", "slow: longer CPU test")


# Canary bands around every ring and split workspace the GPU tests allocate
# through KVRing, checked after each GPU test together with the device error
# word: a kernel that wrote outside its buffers, or a bounded wait or index
# check that fired without the test reading it, fails the test that caused it.
GUARD_BYTES = 64 << 10


@pytest.fixture(autouse=True)
def _device_canaries(request):
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import streaming_attention_block_gb300 as sab

    sab.KVRing.default_guard_bytes = GUARD_BYTES
    sab.guard_watch_begin()
    yield
    bad = sab.guard_watch_end()
    status = sab.get_last_device_error()
    assert bad == 0, f"{bad} canary bytes around ring or workspace memory were overwritten"
    assert status == 0, f"device error word left set: {sab.status_string(status)}"
