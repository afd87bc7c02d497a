"""GPU parity of wo_gemm against the CPU oracle, on the workloads' seeded
inputs: element by element at sizes the oracle finishes in seconds, and on
sampled rows at the workloads' full sizes, in the launch configuration the
bench times.  Tolerance (fp outputs): rel-L2 <= 2e-3 and
max |C - C_ref| <= 1e-2 * max |C_ref| against the fp64 oracle."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from helpers import (DeviceCase, assert_within_tolerance, from_device_bits, sample_rows,
                     to_device_bits)
from weight_only_quantized_fpa_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def wo():
    import weight_only_quantized_fpa_gb300 as w
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w.load_library()
    return w


def _check_full(dc: DeviceCase, what: str):
    C = dc.run()
    torch.cuda.synchronize()
    ref = dc.oracle_rows()
    return assert_within_tolerance(from_device_bits(C), dc.c.act_dtype, ref, what)


def _check_sampled(dc: DeviceCase, what: str, count=64):
    C = dc.run()
    torch.cuda.synchronize()
    rows = sample_rows(dc.c.m, count)
    ref = dc.oracle_rows(rows)
    return assert_within_tolerance(from_device_bits(C)[rows], dc.c.act_dtype, ref, what)


# ------------------------------------------------------ W4 tiny (config 1) --

def test_w4_tiny(wo):
    dc = DeviceCase(inputs.workload_case(1, 0))
    _check_full(dc, "w4 tiny")


# ------------------------------------------------------- small odd shapes --

SMALL = [
    # m, n, k, bits, group, act, zeros, bias
    (1, 64, 64, 8, -1, inputs.F16, False, True),
    (12, 192, 320, 8, -1, inputs.F16, False, True),     # 9-16 rows, a part stage (2 of 4 tiles)
    (16, 320, 576, 8, -1, inputs.BF16, False, False),   # 16 rows, bf16, a part stage
    (7, 128, 1088, 8, -1, inputs.BF16, False, True),    # 1-8 rows, bf16, k split with a part stage
    (3, 192, 320, 8, -1, inputs.F16, False, True),
    (17, 256, 512, 8, -1, inputs.BF16, False, False),
    (5, 320, 1024, 4, 64, inputs.BF16, True, True),
    (16, 128, 640, 4, 64, inputs.F16, True, False),
    (33, 256, 384, 4, 128, inputs.BF16, True, False),
    (2, 128, 512, 4, -1, inputs.BF16, True, True),
    (64, 192, 256, 8, -1, inputs.F16, False, True),
    (65, 128, 256, 4, 64, inputs.BF16, True, True),
    (100, 256, 512, 8, -1, inputs.BF16, False, True),
    (130, 320, 448, 4, 64, inputs.F16, True, False),
    (96, 128, 512, 4, -1, inputs.BF16, True, True),     # per-channel 4-bit, tensor cores
    (80, 256, 1024, 4, 128, inputs.BF16, True, False),  # group 128, tensor cores
    (24, 256, 1024, 4, 128, inputs.F16, True, True),    # group 128, streaming kernel
    (200, 384, 512, 8, -1, inputs.BF16, False, True),   # tensor cores, ragged m and n tiles
    (300, 448, 1024, 4, 64, inputs.BF16, True, True),   # 4-bit, tensor cores, ragged
    (250, 12736, 512, 4, 64, inputs.BF16, True, True),  # 4-bit 256 x 128 tiles, ragged m and n
    (300, 19520, 512, 8, -1, inputs.F16, False, True),  # 128 x 256 tiles, ragged m and n
    (300, 15296, 512, 8, -1, inputs.F16, False, True),  # 256 x 256 tiles (drain helpers), ragged
    (260, 19584, 512, 4, 64, inputs.BF16, True, False), # 4-bit 128 x 256 tiles, ragged
    (300, 15296, 512, 4, 64, inputs.BF16, True, True),  # 4-bit 256 x 256 tiles, ragged
    (200, 320, 6144, 8, -1, inputs.BF16, False, True),  # k split in 2, ragged m and n
    (130, 448, 12288, 4, 64, inputs.BF16, True, True),  # 4-bit, k split in 4, ragged
    (200, 384, 3584, 8, -1, inputs.F16, False, True),   # 128 x 128 tiles, k split in 2, ragged
    (130, 320, 4096, 4, 64, inputs.BF16, True, False),  # 4-bit 128 x 128 tiles, k split in 2
    # one k block: the second MMA issuer of a 128-row tile has nothing to
    # issue and the drain reads only the first partial sum
    (70, 192, 64, 8, -1, inputs.F16, False, True),
    (129, 256, 64, 4, 64, inputs.BF16, True, True),
    (300, 320, 192, 8, -1, inputs.BF16, False, True),   # 3 k blocks: 2 + 1 between the issuers
]


@pytest.mark.parametrize("m,n,k,bits,group,act,zeros,bias", SMALL)
def test_small_shapes(wo, m, n, k, bits, group, act, zeros, bias):
    c = inputs.make_gemm_case(8, m + n + k, m, n, k, bits=bits, group_size=group, act_dtype=act,
                              scale_lo=0.005 if bits == 4 else 0.001,
                              scale_hi=0.02 if bits == 4 else 0.01, with_zeros=zeros,
                              with_bias=bias)
    _check_full(DeviceCase(c), f"m{m} n{n} k{k} w{bits} g{group}")


# 4-bit decode sizes (m <= 16): the persistent kernel's edge cases.  Strips of
# 256 channels (the last one partly past n), stages of 128 codes (a half
# stage at the end when k % 128 == 64), strips cut into pieces across CTAs
# when there are few of them (summed through the workspace by the last
# piece to arrive).  The automatic choice sends these shapes to the cluster
# kernel (it takes the persistent one only for grids wider than a resident
# wave, like the full-size lm_head of the W4 workload);
# test_decode_shapes_on_the_persistent_kernel runs them all again with the
# persistent kernel forced.
PERSISTENT = [
    # m, n, k, bits, group, act, zeros, bias
    (8, 320, 2048, 4, 64, inputs.F16, True, True),       # 8 rows: one activation row block
    (9, 320, 2048, 4, 64, inputs.BF16, True, True),      # 9 rows: two
    (1, 320, 2048, 4, 64, inputs.BF16, True, False),     # one row: tiles spread over columns
    (1, 2112, 4096, 4, 128, inputs.F16, True, True),     # one row, group 128
    (1, 192, 704, 4, -1, inputs.F16, True, True),        # one row, per channel, k % 128 == 64
    (12, 448, 4096, 4, 64, inputs.BF16, True, True),
    (16, 192, 8192, 4, 128, inputs.F16, True, False),    # group 128, few strips, long k
    (1, 704, 1536, 4, 64, inputs.F16, False, True),      # no zeros
    (3, 128, 576, 4, -1, inputs.BF16, True, True),       # per channel, k % 128 == 64
    (1, 64, 11776, 4, 64, inputs.BF16, True, False),     # one strip over many CTAs
    (2, 4160, 192, 4, -1, inputs.F16, True, True),       # many strips, 2 stages each
    (4, 320, 16384, 4, 64, inputs.BF16, True, True),     # long k, few channels
    (7, 2368, 3136, 4, 64, inputs.BF16, True, True),     # k / 64 not a multiple of 8: cluster kernel
]


@pytest.mark.parametrize("m,n,k,bits,group,act,zeros,bias", PERSISTENT)
def test_decode_shapes(wo, m, n, k, bits, group, act, zeros, bias):
    if os.environ.get("WO_DECODE_KERNEL") == "persistent" and (group == -1 or (k // group) % 8 == 0):
        assert wo.gemm_plan(m, n, k, bits, group, act)["kernel"] == "stream_persistent"
    c = inputs.make_gemm_case(14, m + n + k, m, n, k, bits=bits, group_size=group, act_dtype=act,
                              scale_lo=0.005 if bits == 4 else 0.001,
                              scale_hi=0.02 if bits == 4 else 0.01, with_zeros=zeros,
                              with_bias=bias)
    dc = DeviceCase(c)
    _check_full(dc, f"decode m{m} n{n} k{k} w{bits} g{group}")
    C1 = dc.run().clone()
    C2 = dc.run()
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))  # pieces summed in k order


def test_decode_shapes_on_the_persistent_kernel(wo):
    # the decode cases again, in a process whose wo_gemm always takes the
    # persistent kernel where it applies (the choice is read once per process)
    if os.environ.get("WO_DECODE_KERNEL"):
        pytest.skip("already forced")
    env = dict(os.environ, WO_DECODE_KERNEL="persistent")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.abspath(__file__), "-q", "-m", "gpu",
                        "-p", "no:cacheprovider", "-k", "test_decode_shapes and not persistent_kernel"],
                       env=env, capture_output=True, text=True, timeout=600,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert "passed" in r.stdout


@pytest.mark.parametrize("m,n,k,group", [(1, 128, 16384, -1), (4, 256, 16384, 64), (2, 128, 8192, -1)])
def test_w4_nonnegative_activations_long_groups(wo, m, n, k, group):
    # 4-bit codes with bf16 activations that are all >= 0 (as after a gated
    # activation): the decode kernel's group sums then carry the largest
    # activation sums next to the smallest results, per-channel groups span
    # the whole k
    c = inputs.make_gemm_case(8, 400 + m, m, n, k, bits=4, group_size=group, act_dtype=inputs.BF16,
                              scale_lo=0.005, scale_hi=0.02, with_zeros=True, with_bias=True)
    c.A = (c.A & np.uint16(0x7FFF)).astype(c.A.dtype)  # |a|: clear the bf16 sign bits
    _check_full(DeviceCase(c), f"w4 |a| m{m} k{k} g{group}")


# --------------------------------- 4-bit inputs outside fp16's own range --
#
# The tensor-core kernel multiplies 4-bit weights in fp16; its prepass brings
# every output channel's scales and zeros (and bf16 activation rows) into
# fp16's range by powers of two that the epilogue undoes.  These cases would
# overflow fp16 (scales >= 2^13 make (q - 8) * s reach 2^16) or fall into its
# subnormals (scales near 1e-6) without that; activation rows here span more
# than 2^30.  m = 4 runs the weight-streaming kernel, the others the
# tensor-core kernel (k split included).

def _domain_case(m, n, k, act, seed, *, s_lo, s_hi, z_sigma, s_span=0, a_span=0, row_span=0,
                 a_shift=0, group=64, bias=False):
    c = inputs.make_gemm_case(13, seed, m, n, k, bits=4, group_size=group, act_dtype=act,
                              scale_lo=s_lo, scale_hi=s_hi, with_zeros=True, with_bias=bias)
    G = 1 if group in (-1, k) else k // group
    c.zeros = inputs.normal_bits(inputs.rng_for(13, seed, inputs.T_ZERO), c.scales.shape, act,
                                 z_sigma)
    if s_span:  # per group, scales times 2^-u, u uniform in 0..s_span
        u = inputs.rng_for(13, seed, 20).integers(0, s_span + 1, size=(n, G))
        val = oracle.decode(c.scales, act) * np.exp2(-u.astype(np.float64))
        c.scales = inputs.to_bits(val.reshape(c.scales.shape), act)
    if a_span or row_span or a_shift:  # A times 2^u per element, 2^v per row, 2^a_shift
        rng = inputs.rng_for(13, seed, 21)
        u = rng.integers(-a_span, a_span + 1, size=(m, k)) if a_span else 0
        v = rng.integers(-row_span, row_span + 1, size=(m, 1)) if row_span else 0
        val = oracle.decode(c.A, act) * np.exp2(u + v + a_shift)
        c.A = inputs.to_bits(val, act)
    return c


DOMAIN = [
    # m, n, k, act, s_lo, s_hi, z_sigma, extra
    (200, 384, 1024, inputs.BF16, 8192.0, 16384.0, 4096.0, {}),          # (q-8)s beyond 65504
    # fp16 output: A scaled by 2^-10 so that C (about 2^23 otherwise) fits in fp16
    (200, 384, 1024, inputs.F16, 8192.0, 16384.0, 2048.0, dict(a_shift=-10)),
    (4, 384, 1024, inputs.BF16, 8192.0, 16384.0, 4096.0, {}),
    (300, 448, 1024, inputs.BF16, 5e-7, 2e-6, 1e-6, {}),                 # fp16 subnormal scales
    (130, 320, 1024, inputs.F16, 5e-7, 2e-6, 1e-6, {}),
    (4, 320, 1024, inputs.F16, 5e-7, 2e-6, 1e-6, {}),
    (200, 384, 1024, inputs.BF16, 0.005, 0.02, 0.01, dict(a_span=16)),   # rows span 2^32+
    (200, 384, 1024, inputs.BF16, 0.005, 0.02, 0.01, dict(a_span=16, row_span=60, bias=True)),
    (4, 384, 1024, inputs.BF16, 0.005, 0.02, 0.01, dict(a_span=16, row_span=60)),
    (200, 384, 1024, inputs.BF16, 0.005, 0.02, 1e-4, dict(s_span=30)),   # a channel's scales span 2^30
    (130, 448, 12288, inputs.BF16, 8192.0, 16384.0, 4096.0, {}),         # k split in 4
    (96, 128, 512, inputs.BF16, 5e-7, 2e-6, 1e-6, dict(group=-1)),       # per channel
]


@pytest.mark.parametrize("m,n,k,act,s_lo,s_hi,z_sigma,extra", DOMAIN)
def test_w4_inputs_beyond_fp16_range(wo, m, n, k, act, s_lo, s_hi, z_sigma, extra):
    c = _domain_case(m, n, k, act, 500 + m + n + int(np.log2(s_hi) + 64), s_lo=s_lo, s_hi=s_hi,
                     z_sigma=z_sigma, **extra)
    st = _check_full(DeviceCase(c), f"w4 domain m{m} s~{s_hi:g} {extra}")
    assert st["ref_max"] > 0


def test_split_k_long_reduction(wo):
    # few channels and a long k: the k range is split across a cluster of CTAs
    c = inputs.make_gemm_case(8, 77, 4, 64, 18944, bits=8, group_size=-1, act_dtype=inputs.F16,
                              scale_lo=0.001, scale_hi=0.01, with_zeros=False, with_bias=True)
    _check_full(DeviceCase(c), "split-k")


def test_split_k_long_reduction_w4(wo):
    c = inputs.make_gemm_case(8, 78, 3, 128, 13312, bits=4, group_size=64,
                              act_dtype=inputs.BF16, scale_lo=0.005, scale_hi=0.02,
                              with_zeros=True, with_bias=True)
    _check_full(DeviceCase(c), "split-k w4")


# ------------------------------------- 17..64 rows (between the regimes) --
#
# 8-bit weights at 17..64 rows take the swap-AB tensor-core kernel while n
# has at most one block of 128 output channels per SM: the blocks are the
# MMA's rows, the activation rows its columns, and a block's k range is
# split across CTAs to fill the SMs (the splits' fp32 sums added in split
# order by the last split to arrive).  Wider n goes to the m >= 65
# tensor-core kernel.  test_mid_shapes_on_the_other_kernels runs the same
# cases on the streaming and the m >= 65 tensor-core kernels.
MID = [
    # m, n, k, act, bias
    (17, 384, 2048, inputs.F16, True),     # 3 blocks, 8 splits
    (24, 4608, 3584, inputs.BF16, True),
    (33, 256, 4160, inputs.F16, False),    # 65 k blocks: a short last split
    (48, 3584, 3584, inputs.BF16, True),
    (64, 1152, 6144, inputs.F16, True),
    (40, 19456, 1024, inputs.F16, True),   # 152 blocks: no split
    (64, 3584, 18944, inputs.BF16, False),  # long k
    (40, 37888, 1024, inputs.F16, True),   # 296 blocks: the m >= 65 kernel
    (20, 256, 64, inputs.F16, True),       # one k block: one partial accumulator
    (40, 512, 192, inputs.BF16, False),    # 3 k blocks: 2 + 1 between the MMA issuers
]


@pytest.mark.parametrize("m,n,k,act,bias", MID)
def test_mid_shapes(wo, m, n, k, act, bias):
    if not os.environ.get("WO_MID_KERNEL"):
        want = "tensor_core_swap_ab" if n // 128 <= torch.cuda.get_device_properties(0).multi_processor_count \
            else "tensor_core"
        assert wo.gemm_plan(m, n, k, 8, -1, act)["kernel"] == want
    c = inputs.make_gemm_case(15, m + n + k, m, n, k, bits=8, group_size=-1, act_dtype=act,
                              scale_lo=0.001, scale_hi=0.01, with_zeros=False, with_bias=bias)
    dc = DeviceCase(c)
    _check_full(dc, f"mid m{m} n{n} k{k}")
    C1 = dc.run().clone()
    C2 = dc.run()
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))  # splits summed in order


@pytest.mark.parametrize("kernel", ["stream", "tensor_core"])
def test_mid_shapes_on_the_other_kernels(wo, kernel):
    # the same cases in a process whose wo_gemm takes another kernel at
    # 17..64 rows (the choice is read once per process)
    if os.environ.get("WO_MID_KERNEL"):
        pytest.skip("already forced")
    env = dict(os.environ, WO_MID_KERNEL=kernel)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.abspath(__file__), "-q", "-m", "gpu",
                        "-p", "no:cacheprovider", "-k", "test_mid_shapes and not other_kernels"],
                       env=env, capture_output=True, text=True, timeout=600,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert "passed" in r.stdout


@pytest.mark.parametrize("case", range(len(inputs.W8_MID["shapes"])))
def test_w8_mid_full(wo, case):
    dc = DeviceCase(inputs.workload_case(11, case))
    _check_full(dc, dc.c.name)


# ------------------------------------------------ A16W8 decode (config 2) --

@pytest.mark.parametrize("case", range(len(inputs.W8_DECODE["shapes"])))
def test_w8_decode_full(wo, case):
    dc = DeviceCase(inputs.workload_case(2, case))
    _check_full(dc, dc.c.name)


# ---------------------------------------------- A16W8 large m (config 3) --

@pytest.mark.parametrize("case", range(len(inputs.W8_LARGE["shapes"])))
def test_w8_large_m_sampled(wo, case):
    dc = DeviceCase(inputs.workload_case(3, case))
    _check_sampled(dc, dc.c.name)


# ------------------------------------------------- W4 group-64 (config 4) --

@pytest.mark.parametrize("case", range(len(inputs.W4_G64["shapes"])))
def test_w4_g64(wo, case):
    dc = DeviceCase(inputs.workload_case(4, case))
    if dc.c.m == 1:
        _check_full(dc, dc.c.name)
    else:
        _check_sampled(dc, dc.c.name)


# ---------------------------------------------------------- properties -----

@pytest.mark.parametrize("config,case", [(2, 3), (2, 11), (3, 1), (4, 6), (4, 9)])
def test_deterministic_bit_identical(wo, config, case):
    # (4, 9) splits k: the partial sums are added in split order whichever
    # unit arrives last, and the per-tile counters return to zero
    dc = DeviceCase(inputs.workload_case(config, case))
    C1 = dc.run().clone()
    C2 = dc.run().clone()
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


def test_integer_exact_case(wo):
    # integer A in -2..2, codes 126..130, scale 1: exact in fp16 everywhere
    m, n, k = 5, 128, 256
    rng = np.random.default_rng(12)
    Ai = rng.integers(-2, 3, size=(m, k))
    qi = rng.integers(126, 131, size=(n, k))
    A = to_device_bits(Ai.astype(np.float16).view(np.uint16), inputs.F16)
    B = wo.pack(torch.from_numpy(qi.astype(np.uint8)).cuda(), n, k, 8)
    s = to_device_bits(np.full(n, np.float16(1.0).view(np.uint16)), inputs.F16)
    C = wo.gemm(A, B, s, n, k, 8)
    torch.cuda.synchronize()
    ref = (Ai @ (qi - 128).T).astype(np.float16).view(np.uint16)
    assert np.array_equal(from_device_bits(C), ref)


def test_empty_m_is_noop(wo):
    c = inputs.workload_case(1, 0)
    dc = DeviceCase(c)
    A0 = torch.empty((0, c.k), dtype=dc.A.dtype, device="cuda")
    C = dc.run(A=A0)
    assert C.shape == (0, c.n)


def test_output_overwrites_poisoned_buffer(wo):
    dc = DeviceCase(inputs.workload_case(1, 0))
    out = torch.full((1, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    dc.run(out=out)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("m,n,k,bits,group", [(200, 384, 512, 8, -1), (4096, 4096, 1024, 8, -1),
                                                (300, 448, 1024, 4, 64)])
def test_output_16_byte_aligned(wo, m, n, k, bits, group):
    # C 16- but not 32-byte aligned: the tensor-core epilogue stores 16 bytes
    # at a time instead of 32
    c = inputs.make_gemm_case(8, 95 + m, m, n, k, bits=bits, group_size=group, act_dtype=inputs.BF16,
                              scale_lo=0.005 if bits == 4 else 0.001,
                              scale_hi=0.02 if bits == 4 else 0.01, with_zeros=bits == 4,
                              with_bias=True)
    dc = DeviceCase(c)
    buf = torch.empty(m * n + 8, dtype=dc.A.dtype, device="cuda")
    assert buf.data_ptr() % 32 == 0
    out = buf[8:].view(m, n)  # 16 bytes past a 32-byte boundary
    dc.run(out=out)
    torch.cuda.synchronize()
    rows = sample_rows(m, 16)
    assert_within_tolerance(from_device_bits(out)[rows], c.act_dtype, dc.oracle_rows(rows),
                            "16-byte aligned C")


def test_workspace_shared_across_shapes(wo):
    # calls of different kernels and shapes sharing one workspace, twice over:
    # a tensor-core call with a converted-activation scratch region, a
    # cluster-split decode call and a second tensor-core call of another size
    a = DeviceCase(inputs.make_gemm_case(8, 90, 200, 256, 1024, bits=4, group_size=64,
                                         act_dtype=inputs.BF16, scale_lo=0.005, scale_hi=0.02,
                                         with_zeros=True, with_bias=True))
    b = DeviceCase(inputs.make_gemm_case(8, 91, 16, 64, 18944, bits=8, group_size=-1,
                                         act_dtype=inputs.F16, scale_lo=0.001, scale_hi=0.01,
                                         with_zeros=False, with_bias=True))
    c = DeviceCase(inputs.make_gemm_case(8, 92, 96, 512, 512, bits=8, group_size=-1,
                                         act_dtype=inputs.BF16, scale_lo=0.001, scale_hi=0.01,
                                         with_zeros=False, with_bias=False))
    need = max(wo.wo_workspace_size(200, 256, 1024, 64, 4),
               wo.wo_workspace_size(16, 64, 18944, -1, 8),
               wo.wo_workspace_size(96, 512, 512, -1, 8))
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        Ca = a.run(workspace=ws)
        Cb = b.run(workspace=ws)
        Cc = c.run(workspace=ws)
        torch.cuda.synchronize()
        assert_within_tolerance(from_device_bits(Ca), inputs.BF16, a.oracle_rows(), "tc w4")
        assert_within_tolerance(from_device_bits(Cb), inputs.F16, b.oracle_rows(), "decode")
        assert_within_tolerance(from_device_bits(Cc), inputs.BF16, c.oracle_rows(), "tc w8")
    assert wo.wo_check_workspace(ws, ws.numel()) == 0


@pytest.mark.parametrize("m", [1, 16])
def test_chained_calls_keep_stream_order(wo, m):
    # Y = X . W1^T, then X = Y . W2^T on one stream with no sync in between:
    # the second call must read Y only after the first wrote it, and must not
    # overwrite X before the first has read it (the small-m kernel starts
    # early and prefetches weights while the previous kernel finishes)
    n = k = 3584
    c1 = inputs.make_gemm_case(8, 200 + m, m, n, k, bits=8, group_size=-1, act_dtype=inputs.F16,
                               scale_lo=0.001, scale_hi=0.01, with_zeros=False, with_bias=False)
    c2 = inputs.make_gemm_case(8, 300 + m, m, n, k, bits=8, group_size=-1, act_dtype=inputs.F16,
                               scale_lo=0.001, scale_hi=0.01, with_zeros=False, with_bias=False)
    d1, d2 = DeviceCase(c1), DeviceCase(c2)
    X = d1.A.clone()
    Y = torch.empty((m, n), dtype=X.dtype, device="cuda")
    for _ in range(3):
        X.copy_(d1.A)
        wo.gemm(X, d1.B, d1.scales, n, k, 8, out=Y)
        wo.gemm(Y, d2.B, d2.scales, n, k, 8, out=X)
        torch.cuda.synchronize()
        y = from_device_bits(Y)
        assert_within_tolerance(y, inputs.F16, d1.oracle_rows(), "first call")
        ref2 = oracle.gemm(y, inputs.F16, c2.B, c2.scales, None, None, m, n, k, -1, 8)
        assert_within_tolerance(from_device_bits(X), inputs.F16, ref2, "second call")
