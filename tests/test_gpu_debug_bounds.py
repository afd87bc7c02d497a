"""The index-checked debug build on the GPU.  A library compiled with
-DWO_DEBUG_BOUNDS=1 (csrc/wo_bounds.cuh) checks every global index its
kernels compute against the extent of its buffer; a failed check skips the
access and records its site, so a bad index shows up as a status instead of
a memory fault.  It stands in for a memory checker, which these GPUs do not
offer.

test_gpu_suite_under_index_checks builds that library and reruns the GPU
parity suite in a child process that loads it (WO_DEBUG_BOUNDS=1): the
parity assertions still hold, and the conftest there checks after every test
that no index check fired.  In that child, test_bad_permutation_is_reported
hands the act-order gather a permutation with an entry outside [0, k) --
which the gather reads as 0 by contract, in either build -- and expects the
check to report the gather's site."""
import os
import subprocess
import sys

import pytest

import oracle
from helpers import assert_within_tolerance, from_device_bits, to_device_bits, to_device_u8
from weight_only_quantized_fpa_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHILD = os.environ.get("WO_DEBUG_BOUNDS") == "1"


@pytest.fixture(scope="module")
def wo():
    import weight_only_quantized_fpa_gb300 as w
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w.load_library()
    return w


def test_gpu_suite_under_index_checks(wo):
    if CHILD:
        pytest.skip("this is the child run")
    from weight_only_quantized_fpa_gb300 import build
    lib = build.build(debug_bounds=True)
    assert os.path.exists(lib)
    env = dict(os.environ, WO_DEBUG_BOUNDS="1")
    # the tests that start children of their own (kernel overrides) are left
    # out: their kernels are the same ones the rest of the suite runs
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests"), "-q", "-rA", "-m", "gpu",
                        "-p", "no:cacheprovider", "-k",
                        "not on_the_persistent_kernel and not on_the_other_kernels and not under_index_checks"],
                       env=env, capture_output=True, text=True, timeout=1500, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-6000:] + r.stderr[-2000:]
    assert "PASSED tests/test_gpu_debug_bounds.py::test_bad_permutation_is_reported" in r.stdout, \
        r.stdout[-3000:]


def test_normal_build_reports_no_checks(wo):
    if CHILD:
        pytest.skip("the child loads the checked build")
    st, site = wo.wo_debug_bounds()
    assert st == 2 and site == 0  # WO_ERR_UNSUPPORTED


def test_bad_permutation_is_reported(wo):
    if not CHILD:
        pytest.skip("needs the index-checked build (runs in the child of the test above)")
    st, site = wo.wo_debug_bounds()
    assert (st, site) == (0, 0)
    m, n, k, group = 3, 128, 512, 128
    c = inputs.make_gemm_case(12, 77, m, n, k, bits=4, group_size=group, act_dtype=inputs.BF16,
                              scale_lo=0.005, scale_hi=0.02, with_zeros=True, with_bias=False,
                              act_order=True)
    perm_host = wo.act_order_perm(c.g_idx, c.k, c.group_size)
    perm = perm_host.cuda()
    B = wo.pack_act_order(to_device_u8(c.B), perm, n, k, 4)
    torch.cuda.synchronize()
    assert wo.wo_debug_bounds() == (0, 0)  # a valid permutation passes every check
    bad = perm.clone()
    j = 5
    bad[j] = k  # one entry outside [0, k)
    A = to_device_bits(c.A, c.act_dtype)
    s = to_device_bits(c.scales, c.act_dtype)
    z = to_device_bits(c.zeros, c.act_dtype)
    C = wo.gemm_act_order(A, B, bad, s, n, k, 4, group, zeros=z)
    torch.cuda.synchronize()
    st, site = wo.wo_debug_bounds()
    assert st == 6 and site in (0x601, 0x602), (st, hex(site))  # WO_ERR_BOUNDS at the gather
    assert wo.wo_debug_bounds() == (0, 0)  # read once, cleared
    # the skipped read is the documented zero: column j of the gathered A is 0
    A0 = c.A.copy()
    A0[:, perm_host[j].item()] = 0  # the sorted column j held checkpoint column perm[j]
    ref = oracle.gemm_gidx(A0, c.act_dtype, c.B, c.scales, c.zeros, c.g_idx, None, m, n, k, group, 4)
    assert_within_tolerance(from_device_bits(C), c.act_dtype, ref, "bad permutation entry reads 0")
