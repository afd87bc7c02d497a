"""wo_gemm_tc_noalloc, the entry point for callers that cannot allocate device
memory (its scratch is a fixed array inside the library): on the GPU its
output must match wo_gemm's, through the C ABI, on two calls in a row; and it
must refuse problems larger than its built-in scratch without launching.

Kept in a file pytest collects last, so that a failure here comes after every
other test has run; it also passes on its own in a fresh process."""
import numpy as np
import pytest

from helpers import DeviceCase, assert_within_tolerance, from_device_bits
from weight_only_quantized_fpa_gb300 import inputs

torch = pytest.importorskip("torch")


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
def test_noalloc_matches_wo_gemm(wo, m, n, k, bits, group, act, zeros, bias):
    c = inputs.make_gemm_case(7, m + n + k + bits, m, n, k, bits=bits, group_size=group,
                              act_dtype=act, scale_lo=0.005 if bits == 4 else 0.001,
                              scale_hi=0.02 if bits == 4 else 0.01, with_zeros=zeros,
                              with_bias=bias)
    dc = DeviceCase(c)
    ref = dc.run()                    # the existing entry point, with a workspace
    torch.cuda.synchronize()
    ref_bits = from_device_bits(ref)
    lib = wo.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):                # two calls in a row share the scratch
        out = torch.full((m, n), float("nan"), dtype=dc.A.dtype, device="cuda")
        st = lib.wo_gemm_tc_noalloc(dc.A.data_ptr(), dc.B.data_ptr(), dc.scales.data_ptr(),
                                    None if dc.zeros is None else dc.zeros.data_ptr(),
                                    None if dc.bias is None else dc.bias.data_ptr(),
                                    out.data_ptr(), m, n, k, group, bits, act, stream)
        assert st == 0, wo.wo_status_string(st)
        torch.cuda.synchronize()
        got = from_device_bits(out)
        # within tolerance, not bit for bit: for some shapes wo_gemm splits k
        # through its workspace, which the built-in scratch does not do
        assert_within_tolerance(got, act, inputs_to_f64(ref_bits, act), "no-alloc vs wo_gemm")


def inputs_to_f64(bits, act):
    import oracle
    return oracle.decode(bits, act)


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
