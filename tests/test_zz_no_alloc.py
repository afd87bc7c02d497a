"""wo_gemm_tc_noalloc, the entry point for callers that cannot allocate device
memory (its scratch is a fixed array inside the library): on the GPU its
output must match the fp64 oracle within the GEMM tolerance, and wo_gemm's
output (the existing entry point, with a caller workspace) within the same
tolerance, through the C ABI, on two calls in a row; it must refuse
problems larger than its built-in scratch without launching; and a bounded
wait that runs out on the built-in scratch must be reported by
wo_noalloc_check.

Kept in a file pytest collects last, so that a failure here comes after every
other test has run; it also passes on its own in a fresh process."""
import numpy as np
import pytest

import oracle
from helpers import DeviceCase, assert_within_tolerance, from_device_bits
from weight_only_quantized_fpa_gb300 import inputs

torch = pytest.importorskip("torch")

WO_OK, WO_ERR_TIMEOUT = 0, 5


@pytest.fixture(scope="module")
def wo():
    import weight_only_quantized_fpa_gb300 as w
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w.load_library()
    return w


CASES = [
    # m, n, k, bits, group, act, zeros, bias
    (512, 2048, 2048, 4, 64, inputs.BF16, True, False),   # needs the fp16 copy of A
    (200, 512, 1024, 4, 64, inputs.BF16, True, True),
    (300, 768, 512, 8, -1, inputs.F16, False, True),
    (40, 256, 512, 4, 64, inputs.F16, True, False),       # small m still uses the tensor-core kernel
]


@pytest.mark.gpu
@pytest.mark.parametrize("m,n,k,bits,group,act,zeros,bias", CASES)
def test_noalloc_matches_oracle_and_wo_gemm(wo, m, n, k, bits, group, act, zeros, bias):
    c = inputs.make_gemm_case(7, m + n + k + bits, m, n, k, bits=bits, group_size=group,
                              act_dtype=act, scale_lo=0.005 if bits == 4 else 0.001,
                              scale_hi=0.02 if bits == 4 else 0.01, with_zeros=zeros,
                              with_bias=bias)
    dc = DeviceCase(c)
    ref = dc.oracle_rows()            # fp64 oracle, every element
    base = dc.run()                   # the existing entry point, with a workspace
    torch.cuda.synchronize()
    base_f64 = oracle.decode(from_device_bits(base), act)
    lib = wo.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):                # two calls in a row share the scratch
        out = torch.full((m, n), float("nan"), dtype=dc.A.dtype, device="cuda")
        st = lib.wo_gemm_tc_noalloc(dc.A.data_ptr(), dc.B.data_ptr(), dc.scales.data_ptr(),
                                    None if dc.zeros is None else dc.zeros.data_ptr(),
                                    None if dc.bias is None else dc.bias.data_ptr(),
                                    out.data_ptr(), m, n, k, group, bits, act, stream)
        assert st == WO_OK, wo.wo_status_string(st)
        torch.cuda.synchronize()
        got = from_device_bits(out)
        assert_within_tolerance(got, act, ref, "no-alloc vs oracle")
        # and against wo_gemm, within the same tolerance (not bit for bit:
        # for some shapes wo_gemm splits k through its workspace, which the
        # built-in scratch does not do)
        assert_within_tolerance(got, act, base_f64, "no-alloc vs wo_gemm")
    assert wo.wo_noalloc_check() == WO_OK


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch(wo):
    lib = wo.load_library()
    m, n, k = 4096, 256, 4096          # 4-bit with bf16 A: 32 MiB of fp16 copy > 16 MiB
    A = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(n * k // 2, dtype=torch.uint8, device="cuda")
    s = torch.zeros((n, k // 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((m, n), dtype=torch.bfloat16, device="cuda")
    st = lib.wo_gemm_tc_noalloc(A.data_ptr(), B.data_ptr(), s.data_ptr(), None, None,
                                C.data_ptr(), m, n, k, 64, 4, inputs.BF16,
                                torch.cuda.current_stream().cuda_stream)
    assert wo.wo_status_string(st) == "WO_ERR_WORKSPACE"
    torch.cuda.synchronize()
    assert torch.count_nonzero(C) == 0


@pytest.mark.gpu
def test_noalloc_check_reports_a_timeout_on_the_built_in_scratch(wo):
    # a bounded wait that nothing completes gives up after 2 ms and records
    # its code in the built-in scratch's error word; the check reports it
    # once, clears it, and the next no-alloc call is correct
    wo.wo_noalloc_selftest_wait_timeout(2000)
    assert wo.wo_noalloc_check() == WO_ERR_TIMEOUT
    assert wo.wo_noalloc_check() == WO_OK
    m, n, k = 200, 512, 1024
    c = inputs.make_gemm_case(7, 3, m, n, k, bits=4, group_size=64, act_dtype=inputs.BF16,
                              scale_lo=0.005, scale_hi=0.02, with_zeros=True, with_bias=True)
    dc = DeviceCase(c)
    out = torch.empty((m, n), dtype=dc.A.dtype, device="cuda")
    wo.wo_gemm_tc_noalloc(dc.A, dc.B, dc.scales, dc.zeros, dc.bias, out, m, n, k, 64, 4,
                          inputs.BF16)
    torch.cuda.synchronize()
    assert_within_tolerance(from_device_bits(out), inputs.BF16, dc.oracle_rows(), "after timeout")
    assert wo.wo_noalloc_check() == WO_OK
