import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


def read_golden(name):
    """Integer matrix from tests/golden/<name>, skipping '#' comment lines."""
    rows = []
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(t) for t in line.split()])
    return rows


@pytest.fixture(scope="session")
def golden():
    return read_golden


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """Every GPU test must leave the kernels' sticky device status word at FA_OK.  A
    bounded wait that gave up makes its kernel unwind early; this fails the test even
    where the outputs it checks happen to stay within tolerance."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    from exact_tiled_attention_20_gb300 import _lib
    if _lib._lib is None:  # the library was never loaded (the test skipped)
        return
    status = _lib.fa_last_device_status()
    assert status == 0, f"device status {status} ({_lib.fa_status_string(status)}) after the test"
