import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU case")


@pytest.fixture(autouse=True)
def _index_checks_clean(request):
    """Under the index-checked library (WO_DEBUG_BOUNDS=1), every GPU test
    must end with no index check fired (tests that provoke one read and clear
    it themselves)."""
    yield
    if os.environ.get("WO_DEBUG_BOUNDS") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import weight_only_quantized_fpa_gb300 as wo
    if wo._lib is None:  # the test never loaded the library (skipped)
        return
    st, site = wo.wo_debug_bounds()
    assert (st, site) == (0, 0), f"index check at site {site:#x} fired (status {st})"
