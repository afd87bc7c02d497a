"""Failure detection on the GPU without a GPU fault: a bounded mbarrier wait
that nothing completes runs out after a short limit, records an error code in
the workspace header and returns; the host reads it as WO_ERR_TIMEOUT and the
context stays usable for the next call."""
import pytest

from helpers import DeviceCase, assert_within_tolerance, from_device_bits
from weight_only_quantized_fpa_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

WO_OK, WO_ERR_TIMEOUT = 0, 5


@pytest.fixture(scope="module")
def wo():
    import weight_only_quantized_fpa_gb300 as w
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w.load_library()
    return w


def test_bounded_wait_runs_out_and_reports(wo):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    wo.wo_selftest_wait_timeout(ws, ws.numel(), 2000)       # a 2 ms limit
    assert wo.wo_check_workspace(ws, ws.numel()) == WO_ERR_TIMEOUT
    assert wo.wo_check_workspace(ws, ws.numel()) == WO_OK   # the word was cleared


def test_context_usable_after_a_timeout(wo):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    wo.wo_selftest_wait_timeout(ws, ws.numel(), 1000)
    assert wo.wo_check_workspace(ws, ws.numel()) == WO_ERR_TIMEOUT
    dc = DeviceCase(inputs.workload_case(1, 0))
    C = dc.run()
    torch.cuda.synchronize()
    assert_within_tolerance(from_device_bits(C), dc.c.act_dtype, dc.oracle_rows(), "after timeout")
