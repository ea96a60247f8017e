import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libfp8z1.so")
    config.addinivalue_line("markers", "plants_miss: makes the checked kernels skip accesses on purpose")


@pytest.fixture(autouse=True)
def _no_checked_misses(request):
    """Under the checked library (FP8Z1_CHECKED=1), no GPU test may make a
    row-major access outside its param: the checked kernels' skip counter must
    not move (tests marked plants_miss excepted)."""
    if os.environ.get("FP8Z1_CHECKED", "0") in ("", "0") or request.node.get_closest_marker("gpu") is None:
        yield
        return
    from blockwise_fp8_zero_fold_gb300 import fp8z1 as F

    assert F.fp8z1_build_flags() & F.BUILD_CHECKED, "FP8Z1_CHECKED=1 but the release library is loaded"
    before = F.fp8z1_checked_misses()
    yield
    if request.node.get_closest_marker("plants_miss") is None:
        assert F.fp8z1_checked_misses() == before, "a kernel reached outside a param"
