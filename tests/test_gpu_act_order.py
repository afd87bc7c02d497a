"""GPU parity of the GPTQ act-order path (wo_act_order_perm, wo_pack_act_order,
wo_gemm_act_order) against the CPU oracle's gemm_gidx, which indexes the
scales by g_idx[c] directly and permutes nothing.  Tolerance as for wo_gemm:
rel-L2 <= 2e-3 and max |C - C_ref| <= 1e-2 * max |C_ref| against the fp64
oracle; the packed codes are compared bit for bit."""
import numpy as np
import pytest

import oracle
from helpers import (assert_within_tolerance, from_device_bits, sample_rows, to_device_bits,
                     to_device_u8)
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


class ActOrderCase:
    """A GemmCase with a g_idx, uploaded and packed in group-sorted order."""

    def __init__(self, wo, c: inputs.GemmCase):
        self.c = c
        self.perm_host = wo.act_order_perm(c.g_idx, c.k, c.group_size)
        self.perm = self.perm_host.cuda()
        self.A = to_device_bits(c.A, c.act_dtype)
        self.B = wo.pack_act_order(to_device_u8(c.B), self.perm, c.n, c.k, c.bits)
        self.s = to_device_bits(c.scales, c.act_dtype)
        self.z = None if c.zeros is None else to_device_bits(c.zeros, c.act_dtype)
        self.b = None if c.bias is None else to_device_bits(c.bias, c.act_dtype)

    def run(self, wo, A=None, out=None, workspace=None):
        c = self.c
        return wo.gemm_act_order(self.A if A is None else A, self.B, self.perm, self.s, c.n, c.k,
                                 c.bits, c.group_size, zeros=self.z, bias=self.b, out=out,
                                 workspace=workspace)

    def oracle_rows(self, rows=None, A=None):
        c = self.c
        A = c.A if A is None else A
        A = A if rows is None else A[rows]
        return oracle.gemm_gidx(A, c.act_dtype, c.B, c.scales, c.zeros, c.g_idx, c.bias,
                                A.shape[0], c.n, c.k, c.group_size, c.bits)


def _case(m, n, k, group, act, bias, seed, bits=4):
    return inputs.make_gemm_case(12, seed, m, n, k, bits=bits, group_size=group, act_dtype=act,
                                 scale_lo=0.005 if bits == 4 else 0.001,
                                 scale_hi=0.02 if bits == 4 else 0.01, with_zeros=bits == 4,
                                 with_bias=bias, act_order=True)


SHAPES = [
    # m, n, k, group, act, bias
    (1, 256, 1024, 128, inputs.BF16, False),     # streaming kernel, decode
    (1, 512, 2048, 64, inputs.F16, True),
    (5, 320, 1024, 64, inputs.BF16, True),       # ragged m
    (16, 512, 2048, 128, inputs.F16, True),
    (64, 192, 512, 64, inputs.BF16, False),      # last streaming m
    (65, 256, 512, 128, inputs.BF16, True),      # first tensor-core m
    (300, 448, 1024, 64, inputs.BF16, True),     # tensor cores, ragged m and n
    (300, 384, 2048, 128, inputs.F16, False),    # tensor cores, fp16 (no fp16 copy prepass)
    (130, 320, 4096, 128, inputs.BF16, False),   # 128 x 128 tiles, k split in 2
]


@pytest.mark.parametrize("m,n,k,group,act,bias", SHAPES)
def test_act_order_gemm_matches_oracle(wo, m, n, k, group, act, bias):
    c = _case(m, n, k, group, act, bias, seed=m + k // 64)
    ac = ActOrderCase(wo, c)
    C = ac.run(wo)
    torch.cuda.synchronize()
    assert_within_tolerance(from_device_bits(C), act, ac.oracle_rows(), f"act-order m={m}")


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_act_order_is_the_permuted_pack(wo, bits):
    # unpacking the act-order pack gives the row-major codes with columns in
    # the order perm, bit for bit
    n, k, group = 192, 1024, 128
    c = _case(1, n, k, group if bits == 4 else -1, inputs.BF16, False, seed=40 + bits, bits=bits)
    if bits == 8:  # per channel: any channel order is a valid act-order pack
        c.g_idx = np.zeros(k, dtype=np.int32)
        perm = inputs.rng_for(12, 41, 12).permutation(k).astype(np.int32)
    else:
        perm = wo.act_order_perm(c.g_idx, k, group).numpy()
    Bp = wo.pack_act_order(to_device_u8(c.B), torch.from_numpy(perm).cuda(), n, k, bits)
    got = wo.unpack(Bp, n, k, bits).cpu().numpy()
    if bits == 8:
        ref = c.B[:, perm]
    else:
        q = np.empty((n, k), dtype=np.uint8)
        q[:, 0::2] = c.B & 0x0F
        q[:, 1::2] = c.B >> 4
        q = q[:, perm]
        ref = q[:, 0::2] | (q[:, 1::2] << 4)
    assert np.array_equal(got, ref)


def test_in_order_g_idx_equals_plain_gemm_bitwise(wo):
    # g_idx = c // group sorts to the identity: the gathered copy is A itself
    # and the same kernels run, so C is bit-identical to wo_gemm's
    for m in (4, 200):
        c = _case(m, 384, 2048, 128, inputs.BF16, True, seed=50 + m)
        c.g_idx = (np.arange(c.k) // 128).astype(np.int32)
        ac = ActOrderCase(wo, c)
        assert torch.equal(ac.perm_host, torch.arange(c.k, dtype=torch.int32))
        B_plain = wo.pack(to_device_u8(c.B), c.n, c.k, c.bits)
        C1 = ac.run(wo)
        C2 = wo.gemm(ac.A, B_plain, ac.s, c.n, c.k, c.bits, group_size=128, zeros=ac.z, bias=ac.b)
        torch.cuda.synchronize()
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


def test_w8_per_channel_any_order_matches_plain_oracle(wo):
    # 8-bit per channel: one group, so the channel order changes nothing but
    # the summation order
    m, n, k = 3, 256, 1024
    c = _case(m, n, k, -1, inputs.F16, True, seed=60, bits=8)
    assert np.all(c.g_idx == 0)
    perm = torch.from_numpy(inputs.rng_for(12, 61, 12).permutation(k).astype(np.int32)).cuda()
    A = to_device_bits(c.A, c.act_dtype)
    B = wo.pack_act_order(to_device_u8(c.B), perm, n, k, 8)
    s = to_device_bits(c.scales, c.act_dtype)
    b = to_device_bits(c.bias, c.act_dtype)
    C = wo.gemm_act_order(A, B, perm, s, n, k, 8, -1, bias=b)
    torch.cuda.synchronize()
    ref = oracle.gemm(c.A, c.act_dtype, c.B, c.scales, None, c.bias, m, n, k, -1, 8)
    assert_within_tolerance(from_device_bits(C), c.act_dtype, ref, "w8 act-order")


@pytest.mark.parametrize("case", [2, 3, 7, 8])
def test_act_order_workload_sampled(wo, case):
    # the bench workload's full sizes (13312 and 131072 x 2048, group 128) in
    # its launch configuration, on sampled rows
    c = inputs.workload_case(6, case)
    ac = ActOrderCase(wo, c)
    C = ac.run(wo)
    torch.cuda.synchronize()
    rows = sample_rows(c.m)
    assert_within_tolerance(from_device_bits(C)[rows], c.act_dtype, ac.oracle_rows(rows),
                            c.name)


def test_act_order_deterministic_and_reads_fresh_A(wo):
    # the gather reads A only after the previous operation on the stream:
    # A rewritten by the kernel just before the call gives the new result
    c = _case(16, 512, 2048, 128, inputs.BF16, False, seed=70)
    ac = ActOrderCase(wo, c)
    C1 = ac.run(wo).clone()
    C1b = ac.run(wo)
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int16), C1b.view(torch.int16))
    A2_bits = inputs.normal_bits(inputs.rng_for(12, 71, 1), (c.m, c.k), c.act_dtype)
    A2 = to_device_bits(A2_bits, c.act_dtype)
    Adst = torch.empty_like(ac.A)
    Adst.copy_(A2)
    C2 = ac.run(wo, A=Adst)
    torch.cuda.synchronize()
    assert_within_tolerance(from_device_bits(C2), c.act_dtype, ac.oracle_rows(A=A2_bits),
                            "fresh A")


@pytest.mark.parametrize("m", [16, 200])
def test_act_order_workspace_shared_with_plain_gemm(wo, m):
    # the act-order workspace starts with the plain GEMM's (same header and
    # counters) and keeps the gathered A out of the counter area, so one
    # buffer serves both kinds of call in turn, k-split GEMMs included
    c = _case(m, 384, 4096, 128, inputs.BF16, True, seed=80 + m)
    ac = ActOrderCase(wo, c)
    # a k-split GEMM (arrival counters in the workspace) after each act-order call
    sp = inputs.make_gemm_case(12, 90, 200, 320, 6144, bits=8, group_size=-1,
                               act_dtype=inputs.BF16, scale_lo=0.001, scale_hi=0.01,
                               with_zeros=False, with_bias=True)
    need = max(wo.wo_act_order_workspace_size(c.m, c.n, c.k, 128, 4),
               wo.wo_workspace_size(sp.m, sp.n, sp.k, -1, 8))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    sA = to_device_bits(sp.A, sp.act_dtype)
    sB = wo.pack(to_device_u8(sp.B), sp.n, sp.k, 8)
    sS = to_device_bits(sp.scales, sp.act_dtype)
    sb = to_device_bits(sp.bias, sp.act_dtype)
    for _ in range(2):
        C1 = ac.run(wo, workspace=ws)
        C2 = wo.gemm(sA, sB, sS, sp.n, sp.k, 8, bias=sb, workspace=ws)
    torch.cuda.synchronize()
    assert_within_tolerance(from_device_bits(C1), c.act_dtype, ac.oracle_rows(), "shared ws")
    ref_sp = oracle.gemm(sp.A, sp.act_dtype, sp.B, sp.scales, None, sp.bias, sp.m, sp.n, sp.k,
                         -1, 8)
    assert_within_tolerance(from_device_bits(C2), sp.act_dtype, ref_sp, "k split after")
    assert wo.wo_check_workspace(ws, need) == 0


@pytest.mark.parametrize("case", [3, 4, 8, 9])
def test_group128_in_order_workload_sampled(wo, case):
    # the in-order group-128 workload the act-order one is compared with, at
    # full size, through wo_gemm
    from helpers import DeviceCase
    c = inputs.workload_case(7, case)
    dc = DeviceCase(c)
    C = dc.run()
    torch.cuda.synchronize()
    rows = sample_rows(c.m)
    assert_within_tolerance(from_device_bits(C)[rows], c.act_dtype, dc.oracle_rows(rows), c.name)
