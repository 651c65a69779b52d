"""Shared test configuration.

Markers: `gpu` for tests that need a CUDA device (the parity tests proper);
everything else runs on a CPU-only host.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")


@pytest.fixture(autouse=True)
def _no_index_fault(request):
    """After every GPU test: no kernel recorded an out-of-range index.  Only
    the index-checked library (W4A16_LIBRARY=checked) sets that bit, where an
    index check that fails skips the access; the status word persists, so a
    later test would report an earlier one's fault too."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import int4_weight_only_gemv_gb300 as w4
    if w4._LIB is None:
        return
    assert not w4.w4a16_device_status(clear=False) & w4.DEV_INDEX, "a kernel recorded an out-of-range index"
