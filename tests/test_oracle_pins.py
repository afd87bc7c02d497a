"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against something fixed independently:
the packing rule of the vLLM-Omni ``cpu_int4.py`` docstring worked out by hand
(tests/golden), brute-force per-element loops written here, library routines
(numpy float16 casts, numpy float64 matmul, integer matmul), closed forms and
the min/max quantiser invariant of ``cpu_int4.py`` ``quantize_groupwise``.
A plausible slip in the oracle -- a dropped zero term, a wrong code offset or
sign, the nibbles swapped, a transposed operand, a wrong rounding -- fails at
least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from weight_only_quantized_fpa_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F16, BF16 = oracle.F16, oracle.BF16


# ----------------------------------------------------------------- helpers --

def _read_nibble_golden():
    cases = []
    with open(os.path.join(GOLDEN, "nibble_rule.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            codes, hexes = line.split("|")
            cases.append(([int(c) for c in codes.split()],
                          [int(h, 16) for h in hexes.split()]))
    return cases


def _np_half_value(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _np_bf16_value(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _value(bits, dtype):
    return _np_half_value(bits) if dtype == F16 else _np_bf16_value(bits)


def _test_unpack(B, n, k, bits):
    """Codes from row-major storage, written independently of the oracle."""
    if bits == 8:
        return B.reshape(n, k).astype(np.int64)
    q = np.empty((n, k), dtype=np.int64)
    q[:, 0::2] = B & 0x0F
    q[:, 1::2] = B >> 4
    return q


def _test_dequant_f32(B, scales, zeros, n, k, group_size, bits, dtype):
    """fp32 dequantisation written here: (q - off) * s + z, product and sum
    rounded separately in fp32."""
    q = _test_unpack(B, n, k, bits)
    off = 8 if bits == 4 else 128
    g = k if group_size in (-1, k) else group_size
    s = _value(scales, dtype).reshape(n, -1).astype(np.float32)
    s = np.repeat(s, g, axis=1)
    w = (q - off).astype(np.float32) * s
    if zeros is not None:
        z = np.repeat(_value(zeros, dtype).reshape(n, -1).astype(np.float32), g, axis=1)
        w = (w + z).astype(np.float32)
    return w


# ------------------------------------------------------- number formats ----

def test_half_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, F16)
    ref = _np_half_value(bits)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bf16_decode_all_patterns_match_fp32_upper_half():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, BF16)
    ref = _np_bf16_value(bits)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_half_encode_matches_numpy_cast():
    # numpy's float64 -> float16 cast rounds to nearest even in one step
    rng = np.random.default_rng(7)
    x = rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 17, 200000))
    x = np.concatenate([x, [0.0, -0.0, 65504.0, 65519.99, 65520.0, 2.0**-24,
                            2.0**-25, 3 * 2.0**-26, 2.0**-14, -(2.0**-14) * (1 - 2**-11)]])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert (oracle.round_to(x, F16) == ref).all()


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80), (-2.0, 0xC000),
    (1.0 + 2.0**-8, 0x3F80),          # tie -> even (down)
    (1.0 + 3 * 2.0**-8, 0x3F82),      # tie -> even (up)
    (1.0 + 2.0**-8 + 2.0**-40, 0x3F81),  # just above the tie
    (3.3895313892515355e38, 0x7F7F),  # largest finite bf16
    (3.4e38, 0x7F80),                 # rounds past the largest finite -> inf
    (2.0**-133, 0x0001),              # smallest subnormal
    (2.0**-134, 0x0000),              # tie with zero -> even (zero)
    (1.5 * 2.0**-134, 0x0001),
    (2.0**-126, 0x0080),              # smallest normal
])
def test_bf16_encode_special_values(x, bits):
    # worked out from the bfloat16 format: 1 sign, 8 exponent (bias 127), 7 fraction bits
    assert oracle.to_bf16_bits(x) == bits


def test_bf16_encode_matches_fp32_rounding():
    # for fp32-representable inputs, rounding fp32 -> bf16 is a single rounding
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(200000) * np.exp2(rng.uniform(-60, 60, 200000))).astype(np.float32)
    ref = inputs.f32_to_bf16_bits(x)
    assert (oracle.round_to(x.astype(np.float64), BF16) == ref).all()


# ------------------------------------------------------------- packing -----

@pytest.mark.parametrize("case", range(len(_read_nibble_golden())))
def test_nibble_rule_golden(case):
    codes, expect = _read_nibble_golden()[case]
    q = np.array([codes], dtype=np.int32)
    packed = oracle.pack_nibbles(q)
    assert packed.tolist() == [expect]
    back = oracle.unpack_codes(np.array([expect], dtype=np.uint8), 1, len(codes), 4)
    assert back.tolist() == [codes]


def test_nibble_rule_index_pattern_brute_force():
    # "pack an index pattern, read back where each nibble landed"
    n, k = 5, 24
    q = np.array([[(7 * r + 3 * c) % 16 for c in range(k)] for r in range(n)], dtype=np.int32)
    packed = oracle.pack_nibbles(q)
    for r in range(n):
        for j in range(k // 2):
            assert packed[r, j] == (int(q[r, 2 * j]) | (int(q[r, 2 * j + 1]) << 4))


@pytest.mark.parametrize("n,k", [(13312, 2048), (2048, 6656), (3072, 2048), (256, 512)])
def test_nibble_round_trip_shapes(n, k):
    rng = np.random.default_rng(n + k)
    B = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    q = oracle.unpack_codes(B, n, k, 4)
    assert q.min() >= 0 and q.max() <= 15
    assert np.array_equal(oracle.pack_nibbles(q), B)


def test_int8_unpack_is_identity():
    rng = np.random.default_rng(3)
    B = rng.integers(0, 256, size=(7, 64), dtype=np.uint8)
    assert np.array_equal(oracle.unpack_codes(B, 7, 64, 8), B.astype(np.int32))


def test_pack_rejects_out_of_range_codes():
    with pytest.raises(ValueError):
        oracle.pack_nibbles(np.array([[16, 0]], dtype=np.int32))


# ------------------------------------------------------- dequantisation -----

def _quantize_groupwise_f32(w, group):
    """Min/max 4-bit quantiser of cpu_int4.py quantize_groupwise, in fp32:
    scale = (max - min)/15 (clamped at 1e-9), zero = min + 8*scale,
    q = round((w - min)/scale) clamped to 0..15."""
    n, k = w.shape
    wf = w.astype(np.float32).reshape(n, k // group, group)
    wmin, wmax = wf.min(axis=-1), wf.max(axis=-1)
    scale = (np.maximum(wmax - wmin, np.float32(1e-9)) / np.float32(15.0)).astype(np.float32)
    zero = (wmin + np.float32(8.0) * scale).astype(np.float32)
    q = np.clip(np.round((wf - wmin[..., None]) / scale[..., None]), 0, 15).astype(np.int32)
    return q.reshape(n, k), scale, zero, wmin, wmax


def test_quantizer_invariant_exact_values():
    # min = -0.5, max = 1.375: scale = 0.125 and zero = 0.5 are exact in bf16,
    # so (q - 8)*scale + zero must give the extremes exactly at q = 0 and 15.
    w = np.linspace(-0.5, 1.375, 64, dtype=np.float32)[None, :]
    q, scale, zero, wmin, wmax = _quantize_groupwise_f32(w, 64)
    assert scale[0, 0] == np.float32(0.125) and zero[0, 0] == np.float32(0.5)
    assert q[0, 0] == 0 and q[0, -1] == 15
    B = oracle.pack_nibbles(q)
    s_bits = inputs.f32_to_bf16_bits(scale.reshape(1, 1))
    z_bits = inputs.f32_to_bf16_bits(zero.reshape(1, 1))
    deq = oracle.dequant(B, s_bits, z_bits, 1, 64, 64, 4, BF16)
    assert deq[0, 0] == np.float32(-0.5)
    assert deq[0, -1] == np.float32(1.375)


def test_quantizer_invariant_random_groups():
    # with fp16-stored scale/zero the extremes come back within fp16 rounding;
    # a wrong offset or sign convention is off by a whole multiple of scale
    rng = np.random.default_rng(11)
    w = rng.standard_normal((32, 256)).astype(np.float32)
    q, scale, zero, wmin, wmax = _quantize_groupwise_f32(w, 64)
    B = oracle.pack_nibbles(q)
    s_bits = scale.astype(np.float16).view(np.uint16)
    z_bits = zero.astype(np.float16).view(np.uint16)
    deq = oracle.dequant(B, s_bits, z_bits, 32, 256, 64, 4, F16).reshape(32, 4, 64)
    qg = q.reshape(32, 4, 64)
    tol = 2.0**-9 * (np.abs(wmin) + np.abs(wmax)) + 2.0**-9 * 8 * scale
    lo = np.where(qg == 0, deq, np.inf).min(axis=-1)
    hi = np.where(qg == 15, deq, -np.inf).max(axis=-1)
    assert np.all(np.abs(lo - wmin) <= tol)
    assert np.all(np.abs(hi - wmax) <= tol)
    # and every code reproduces its grid point (q - 8)*scale + zero
    grid = (qg - 8).astype(np.float64) * s_bits.view(np.float16).astype(np.float64)[..., None] \
        + z_bits.view(np.float16).astype(np.float64)[..., None]
    assert np.allclose(deq, grid, rtol=2.0**-22, atol=2.0**-30)


@pytest.mark.parametrize("bits,group,dtype,zeros", [
    (4, 64, BF16, True), (4, 128, F16, True), (4, -1, BF16, True),
    (8, -1, F16, False), (8, -1, BF16, True), (8, 64, F16, False)])
def test_dequant_matches_independent_dequant(bits, group, dtype, zeros):
    n, k = 24, 256
    c = inputs.make_gemm_case(9, bits + group % 7, 1, n, k, bits=bits, group_size=group,
                              act_dtype=dtype, scale_lo=0.005, scale_hi=0.02,
                              with_zeros=zeros, with_bias=False)
    got = oracle.dequant(c.B, c.scales, c.zeros, n, k, group, bits, dtype)
    ref = _test_dequant_f32(c.B, c.scales, c.zeros, n, k, group, bits, dtype)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ GEMM -----

def _brute_force_gemm(c):
    """Per-element triple loop in Python floats (fp64), ascending k."""
    q = _test_unpack(c.B, c.n, c.k, c.bits).tolist()
    off = 8 if c.bits == 4 else 128
    g = c.k if c.group_size in (-1, c.k) else c.group_size
    A = _value(c.A, c.act_dtype).reshape(c.m, c.k).tolist()
    S = _value(c.scales, c.act_dtype).reshape(c.n, -1).tolist()
    Z = None if c.zeros is None else _value(c.zeros, c.act_dtype).reshape(c.n, -1).tolist()
    bias = None if c.bias is None else _value(c.bias, c.act_dtype).tolist()
    out = [[0.0] * c.n for _ in range(c.m)]
    for j in range(c.n):
        w = []
        for kk in range(c.k):
            prod = float(np.float32(q[j][kk] - off) * np.float32(S[j][kk // g]))
            if Z is not None:
                prod = float(np.float32(prod) + np.float32(Z[j][kk // g]))
            w.append(prod)
        for i in range(c.m):
            acc = 0.0
            for kk in range(c.k):
                acc += A[i][kk] * w[kk]
            if bias is not None:
                acc += bias[j]
            out[i][j] = acc
    return np.array(out)


@pytest.mark.parametrize("m,n,k,bits,group,dtype,zeros,bias", [
    (1, 16, 128, 4, 64, BF16, True, False),
    (2, 24, 192, 4, 64, F16, True, True),
    (3, 64, 256, 8, -1, F16, False, True),
    (3, 8, 64, 8, -1, BF16, True, False),
    (1, 32, 256, 4, 256, BF16, True, True),
])
def test_gemm_brute_force(m, n, k, bits, group, dtype, zeros, bias):
    c = inputs.make_gemm_case(9, m + n + k, m, n, k, bits=bits, group_size=group,
                              act_dtype=dtype, scale_lo=0.005, scale_hi=0.02,
                              with_zeros=zeros, with_bias=bias)
    got = oracle.gemm(c.A, dtype, c.B, c.scales, c.zeros, c.bias, m, n, k, group, bits)
    ref = _brute_force_gemm(c)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("config,case", [(1, 0), (2, 1), (4, 0)])
def test_gemm_matches_library_matmul(config, case):
    c = inputs.workload_case(config, case)
    if c.n * c.k > 20_000_000:
        pytest.skip("too large for a CPU pin")
    got = oracle.gemm(c.A, c.act_dtype, c.B, c.scales, c.zeros, c.bias, c.m, c.n, c.k,
                      c.group_size, c.bits)
    w = _test_dequant_f32(c.B, c.scales, c.zeros, c.n, c.k, c.group_size, c.bits,
                          c.act_dtype).astype(np.float64)
    A = _value(c.A, c.act_dtype).reshape(c.m, c.k)
    ref = A @ w.T
    if c.bias is not None:
        ref = ref + _value(c.bias, c.act_dtype)[None, :]
    assert np.allclose(got, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())


def test_gemm_closed_form_w4_neutral_codes():
    # every code 8 and zero 0: every weight is 0, so C = 0 exactly
    m, n, k = 3, 32, 128
    A = inputs.normal_bits(np.random.default_rng(1), (m, k), BF16)
    B = np.full((n, k // 2), 0x88, dtype=np.uint8)
    s = inputs.uniform_bits(np.random.default_rng(2), (n, k // 64), BF16, 0.005, 0.02)
    z = np.zeros((n, k // 64), dtype=np.uint16)
    C = oracle.gemm(A, BF16, B, s, z, None, m, n, k, 64, 4)
    assert np.all(C == 0.0)


def test_gemm_closed_form_w4_zero_only():
    # every code 8: C[i][j] = sum_g z[j][g] * (sum of A over group g)
    m, n, k = 2, 16, 192
    rng = np.random.default_rng(5)
    A = inputs.normal_bits(rng, (m, k), F16)
    B = np.full((n, k // 2), 0x88, dtype=np.uint8)
    s = inputs.uniform_bits(rng, (n, 3), F16, 0.005, 0.02)
    z = inputs.normal_bits(rng, (n, 3), F16, 0.01)
    C = oracle.gemm(A, F16, B, s, z, None, m, n, k, 64, 4)
    Av = _np_half_value(A).reshape(m, 3, 64).sum(axis=-1)
    ref = Av @ _np_half_value(z).reshape(n, 3).T
    assert np.allclose(C, ref, rtol=1e-12, atol=1e-14)


def test_gemm_closed_form_w8_neutral_codes_give_bias():
    m, n, k = 4, 64, 128
    rng = np.random.default_rng(6)
    A = inputs.normal_bits(rng, (m, k), F16)
    B = np.full((n, k), 128, dtype=np.uint8)
    s = inputs.uniform_bits(rng, (n,), F16, 0.001, 0.01)
    bias = inputs.normal_bits(rng, (n,), F16, 0.1)
    C = oracle.gemm(A, F16, B, s, None, bias, m, n, k, -1, 8)
    assert np.array_equal(C, np.broadcast_to(_np_half_value(bias), (m, n)))


@pytest.mark.parametrize("bits", [4, 8])
def test_gemm_one_hot_rows_pick_weight_columns(bits):
    # A = e_c picks column c of the dequantised weight: C[:, j] = w[j][c]
    n, k = 32, 128
    c = inputs.make_gemm_case(9, 40 + bits, 1, n, k, bits=bits, group_size=64 if bits == 4 else -1,
                              act_dtype=BF16, scale_lo=0.005, scale_hi=0.02,
                              with_zeros=bits == 4, with_bias=False)
    one = inputs.to_bits(np.array([1.0]), BF16)[0]
    cols = [0, 1, 63, 64, 127]
    A = np.zeros((len(cols), k), dtype=np.uint16)
    for i, col in enumerate(cols):
        A[i, col] = one
    C = oracle.gemm(A, BF16, c.B, c.scales, c.zeros, None, len(cols), n, k, c.group_size, bits)
    q = _test_unpack(c.B, n, k, bits)
    off = 8 if bits == 4 else 128
    s = _np_bf16_value(c.scales).reshape(n, -1)
    z = None if c.zeros is None else _np_bf16_value(c.zeros).reshape(n, -1)
    for i, col in enumerate(cols):
        g = col // 64 if bits == 4 else 0
        w = np.float32(q[:, col] - off) * s[:, g].astype(np.float32)
        if z is not None:
            w = (w + z[:, g].astype(np.float32)).astype(np.float32)
        assert np.array_equal(C[i], w.astype(np.float64))


def _read_embed_golden():
    cases = []
    with open(os.path.join(GOLDEN, "embed_rows.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, group, dt, hidden, codes, sc, zc, idx, row = [x.strip() for x in line.split("|")]
            cases.append((int(bits), int(group), F16 if dt == "f16" else BF16, int(hidden),
                          [int(x) for x in codes.split()], [float(x) for x in sc.split()],
                          None if zc == "-" else [float(x) for x in zc.split()], int(idx),
                          [float(x) for x in row.split()]))
    return cases


@pytest.mark.parametrize("case", range(len(_read_embed_golden())))
def test_embed_golden(case):
    # hand-worked rows (tests/golden/embed_rows.txt): dequantisation, the
    # single rounding (two ties to even) and the zero row of an id out of range
    bits, group, dt, hidden, codes, sc, zc, idx, expect = _read_embed_golden()[case]
    q = np.array(codes, dtype=np.uint8)
    vocab = q.size // hidden
    q = q.reshape(vocab, hidden)
    B = q if bits == 8 else (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    s = inputs.to_bits(np.array(sc), dt)
    z = None if zc is None else inputs.to_bits(np.array(zc), dt)
    assert np.array_equal(_value(s, dt), np.array(sc))  # the inputs are exact in dt
    got = oracle.embed(np.array([idx], dtype=np.int32), B, s, z, vocab, hidden, group, bits, dt)
    assert np.array_equal(_value(got[0], dt), np.array(expect))


@pytest.mark.parametrize("bits,group,dtype", [(4, 64, BF16), (8, -1, F16), (4, -1, F16)])
def test_embed_rows_are_identity_gemm_columns(bits, group, dtype):
    # A = I_k gives C[i, j] = w[j][i]: column id of that product, rounded
    # once, is embedding row id; ids out of range give zero rows
    vocab, k = 64, 128
    c = inputs.make_gemm_case(9, 50 + bits, 1, vocab, k, bits=bits, group_size=group,
                              act_dtype=dtype, scale_lo=0.005, scale_hi=0.02,
                              with_zeros=bits == 4, with_bias=False)
    one = inputs.to_bits(np.array([1.0]), dtype)[0]
    eye = np.zeros((k, k), dtype=np.uint16)
    eye[np.arange(k), np.arange(k)] = one
    C = oracle.gemm(eye, dtype, c.B, c.scales, c.zeros, None, k, vocab, k, group, bits)
    ids = np.array([0, 5, 15, 16, 63, -1, 64, 17], dtype=np.int32)
    got = oracle.embed(ids, c.B, c.scales, c.zeros, vocab, k, group, bits, dtype)
    for t, i in enumerate(ids):
        if 0 <= i < vocab:
            assert np.array_equal(got[t], oracle.round_to(C[:, i], dtype))
        else:
            assert not got[t].any()


def test_gemm_integer_exact():
    # integer A in -2..2, int8 codes 126..130 (q - 128 in -2..2), scale 1:
    # every partial sum is a small integer, so C equals the integer matmul
    m, n, k = 5, 48, 256
    rng = np.random.default_rng(12)
    Ai = rng.integers(-2, 3, size=(m, k))
    qi = rng.integers(126, 131, size=(n, k))
    A = Ai.astype(np.float16).view(np.uint16)
    B = qi.astype(np.uint8)
    s = np.full((n,), np.float16(1.0).view(np.uint16), dtype=np.uint16)
    C = oracle.gemm(A, F16, B, s, None, None, m, n, k, -1, 8)
    assert np.array_equal(C, (Ai @ (qi - 128).T).astype(np.float64))


def test_gemm_is_linear_in_A():
    c = inputs.workload_case(1, 0)
    C1 = oracle.gemm(c.A, BF16, c.B, c.scales, c.zeros, None, c.m, c.n, c.k, 64, 4)
    A2 = inputs.to_bits(2.0 * _np_bf16_value(c.A), BF16)   # exact doubling
    C2 = oracle.gemm(A2, BF16, c.B, c.scales, c.zeros, None, c.m, c.n, c.k, 64, 4)
    assert np.array_equal(C2, 2.0 * C1)


def test_gemm_thread_count_does_not_change_result():
    c = inputs.workload_case(1, 0)
    C1 = oracle.gemm(c.A, BF16, c.B, c.scales, c.zeros, None, c.m, c.n, c.k, 64, 4, nthreads=1)
    C4 = oracle.gemm(c.A, BF16, c.B, c.scales, c.zeros, None, c.m, c.n, c.k, 64, 4, nthreads=5)
    assert np.array_equal(C1, C4)


def test_gemm_output_rounding_matches_numpy_half_cast():
    c = inputs.workload_case(2, 1)
    c = inputs.make_gemm_case(2, 1, 2, 256, 512, bits=8, group_size=-1, act_dtype=F16,
                              scale_lo=0.001, scale_hi=0.01, with_zeros=False, with_bias=True)
    C = oracle.gemm(c.A, F16, c.B, c.scales, None, c.bias, c.m, c.n, c.k, -1, 8)
    assert np.array_equal(oracle.round_to(C, F16), C.astype(np.float16).view(np.uint16))


def test_gemm_rejects_bad_group():
    c = inputs.workload_case(1, 0)
    with pytest.raises(ValueError):
        oracle.gemm(c.A, BF16, c.B, c.scales, c.zeros, None, c.m, c.n, c.k, 100, 4)


# ------------------------------------------------- act-order (GPTQ g_idx) ---

def _permute_codes(B, n, k, bits, perm):
    """Row-major codes with input channel j taken from channel perm[j]."""
    q = _test_unpack(B, n, k, bits)[:, perm]
    if bits == 8:
        return np.ascontiguousarray(q.astype(np.uint8))
    q = q.astype(np.uint8)
    return np.ascontiguousarray(q[:, 0::2] | (q[:, 1::2] << 4))


def _gidx_case(seed, m, n, k, group, dtype=BF16, bias=False):
    c = inputs.make_gemm_case(11, seed, m, n, k, bits=4, group_size=group, act_dtype=dtype,
                              scale_lo=0.005, scale_hi=0.02, with_zeros=True, with_bias=bias)
    g = inputs.act_order_g_idx(inputs.rng_for(11, seed, inputs.T_GIDX), k, group)
    return c, g


@pytest.mark.parametrize("group,dtype", [(64, BF16), (128, F16)])
def test_gidx_in_order_equals_grouped_gemm(group, dtype):
    # g_idx[c] = c // group (GPTQ without act-order, or static groups) is the
    # plain group-wise GEMM, bit for bit
    m, n, k = 3, 32, 512
    c, _ = _gidx_case(1 + group, m, n, k, group, dtype, bias=True)
    g = (np.arange(k) // group).astype(np.int32)
    got = oracle.gemm_gidx(c.A, dtype, c.B, c.scales, c.zeros, g, c.bias, m, n, k, group, 4)
    ref = oracle.gemm(c.A, dtype, c.B, c.scales, c.zeros, c.bias, m, n, k, group, 4)
    assert np.array_equal(got, ref)
    assert np.array_equal(oracle.dequant_gidx(c.B, c.scales, c.zeros, g, n, k, group, 4, dtype),
                          oracle.dequant(c.B, c.scales, c.zeros, n, k, group, 4, dtype))


def test_gidx_brute_force():
    m, n, k, group = 2, 8, 128, 64
    c, g = _gidx_case(2, m, n, k, group, BF16, bias=True)
    q = _test_unpack(c.B, n, k, 4).tolist()
    A = _value(c.A, BF16).reshape(m, k).tolist()
    S = _value(c.scales, BF16).reshape(n, -1).tolist()
    Z = _value(c.zeros, BF16).reshape(n, -1).tolist()
    bias = _value(c.bias, BF16).tolist()
    ref = np.zeros((m, n))
    for j in range(n):
        w = [float(np.float32(np.float32(q[j][kk] - 8) * np.float32(S[j][g[kk]]))
                   + np.float32(Z[j][g[kk]])) for kk in range(k)]
        for i in range(m):
            acc = 0.0
            for kk in range(k):
                acc += A[i][kk] * w[kk]
            ref[i, j] = acc + bias[j]
    got = oracle.gemm_gidx(c.A, BF16, c.B, c.scales, c.zeros, g, c.bias, m, n, k, group, 4)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gidx_is_invariant_under_channel_permutation():
    # reordering the input channels of A, B and g_idx together is the same
    # sum in another order
    m, n, k, group = 4, 48, 384, 64
    c, g = _gidx_case(3, m, n, k, group, BF16)
    pi = inputs.rng_for(11, 3, 12).permutation(k)
    Ap = np.ascontiguousarray(c.A.reshape(m, k)[:, pi])
    Bp = _permute_codes(c.B, n, k, 4, pi)
    got = oracle.gemm_gidx(Ap, BF16, Bp, c.scales, c.zeros, g[pi], None, m, n, k, group, 4)
    ref = oracle.gemm_gidx(c.A, BF16, c.B, c.scales, c.zeros, g, None, m, n, k, group, 4)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gidx_sorted_by_group_is_grouped_gemm():
    # sorting the channels by group (stable) makes every group contiguous, so
    # the act-order GEMM becomes the plain group-wise GEMM of the sorted
    # operands
    m, n, k, group = 3, 32, 512, 128
    c, g = _gidx_case(4, m, n, k, group, F16, bias=True)
    sigma = np.argsort(g, kind="stable")
    As = np.ascontiguousarray(c.A.reshape(m, k)[:, sigma])
    Bs = _permute_codes(c.B, n, k, 4, sigma)
    ref = oracle.gemm(As, F16, Bs, c.scales, c.zeros, c.bias, m, n, k, group, 4)
    got = oracle.gemm_gidx(c.A, F16, c.B, c.scales, c.zeros, g, c.bias, m, n, k, group, 4)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gidx_channel_reads_only_its_own_group():
    # A = e_c: the output depends on the scale and zero of group g_idx[c]
    # and on no other group's
    m, n, k, group = 1, 16, 256, 64
    c, g = _gidx_case(5, m, n, k, group, BF16)
    G = k // group
    one = inputs.to_bits(np.array([1.0]), BF16)[0]
    two = inputs.to_bits(np.array([2.0]), BF16)[0]
    for col in (0, 77, 255):
        A = np.zeros((1, k), dtype=np.uint16)
        A[0, col] = one
        base = oracle.gemm_gidx(A, BF16, c.B, c.scales, c.zeros, g, None, 1, n, k, group, 4)
        for gg in range(G):
            s2 = c.scales.reshape(n, G).copy()
            s2[:, gg] = two
            z2 = c.zeros.reshape(n, G).copy()
            z2[:, gg] = two
            C2 = oracle.gemm_gidx(A, BF16, c.B, s2, z2, g, None, 1, n, k, group, 4)
            assert np.array_equal(C2, base) == (gg != g[col])


def _read_gemm_golden():
    cases = []
    with open(os.path.join(GOLDEN, "gemm_worked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, group, q, sc, zc, a, b, c = [p.strip() for p in line.split("|")]
            cases.append((int(bits), int(group), [int(x) for x in q.split()],
                          [float(x) for x in sc.split()],
                          None if zc == "-" else [float(x) for x in zc.split()],
                          [float(x) for x in a.split()], None if b == "-" else float(b),
                          float(c)))
    return cases


@pytest.mark.parametrize("case", range(len(_read_gemm_golden())))
def test_gemm_golden(case):
    bits, group, q, sc, zc, a, bias, expect = _read_gemm_golden()[case]
    k = len(q)
    if bits == 8:
        B = np.array([q], dtype=np.uint8)
    else:
        B = np.array([[q[2 * j] | (q[2 * j + 1] << 4) for j in range(k // 2)]], dtype=np.uint8)
    bf = lambda v: inputs.to_bits(np.array(v, dtype=np.float64), BF16)  # noqa: E731
    C = oracle.gemm(bf([a]), BF16, B, bf([sc]), None if zc is None else bf([zc]),
                    None if bias is None else bf([bias]), 1, 1, k, group, bits)
    assert C[0, 0] == expect


def _read_act_order_golden():
    cases = []
    with open(os.path.join(GOLDEN, "act_order_gemm.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            group, gi, q, sc, zc, a, c = [p.strip() for p in line.split("|")]
            cases.append((int(group), [int(x) for x in gi.split()], [int(x) for x in q.split()],
                          [float(x) for x in sc.split()], [float(x) for x in zc.split()],
                          [float(x) for x in a.split()], float(c)))
    return cases


@pytest.mark.parametrize("case", range(len(_read_act_order_golden())))
def test_gidx_golden(case):
    group, gi, q, sc, zc, a, expect = _read_act_order_golden()[case]
    k = len(q)
    B = np.array([[q[2 * j] | (q[2 * j + 1] << 4) for j in range(k // 2)]], dtype=np.uint8)
    bits = lambda v: inputs.to_bits(np.array(v, dtype=np.float64), BF16)  # noqa: E731
    C = oracle.gemm_gidx(bits([a]), BF16, B, bits([sc]), bits([zc]), np.array(gi, np.int32),
                         None, 1, 1, k, group, 4)
    assert C[0, 0] == expect


def test_gidx_rejects_out_of_range_group():
    m, n, k, group = 1, 16, 128, 64
    c, g = _gidx_case(6, m, n, k, group)
    bad = g.copy()
    bad[5] = k // group
    with pytest.raises(ValueError):
        oracle.gemm_gidx(c.A, BF16, c.B, c.scales, c.zeros, bad, None, m, n, k, group, 4)
    bad[5] = -1
    with pytest.raises(ValueError):
        oracle.gemm_gidx(c.A, BF16, c.B, c.scales, c.zeros, bad, None, m, n, k, group, 4)


# -------------------------------------------------------------------- MoE ---

def test_route_ties_go_to_lower_expert():
    logits = np.array([[0.5, 2.0, 2.0, -1.0],
                       [1.0, 1.0, 1.0, 1.0],
                       [-3.0, 0.0, 7.0, 0.0]], dtype=np.float32)
    ids, w = oracle.moe_route(logits, 2)
    assert ids.tolist() == [[1, 2], [0, 1], [2, 1]]
    # weights are softmax probabilities over all experts at the chosen ids
    for t in range(3):
        ex = np.exp(logits[t].astype(np.float64) - logits[t].max())
        p = ex / ex.sum()
        assert np.allclose(w[t], p[ids[t]], rtol=1e-15)


def test_route_renormalize_sums_to_one():
    logits = np.random.default_rng(3).standard_normal((50, 64)).astype(np.float32)
    ids, w = oracle.moe_route(logits, 2, renormalize=True)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=1e-15)
    ids2, w2 = oracle.moe_route(logits, 2, renormalize=False)
    assert np.array_equal(ids, ids2)
    assert np.all(w2[:, 0] >= w2[:, 1])


def _brute_force_moe(c, tokens, dtype):
    """Dense per-token MoE written here, numpy fp64 matmuls, fp16 h rounding
    through numpy's float16 cast."""
    H, I = c.H, c.I
    A = _value(c.A, dtype).reshape(c.T, H)
    out = np.zeros((len(tokens), H))
    for si, t in enumerate(tokens):
        lg = c.logits[t]
        order = sorted(range(c.E), key=lambda e: (-float(lg[e]), e))[:c.topk]
        ex = np.exp(lg.astype(np.float64) - lg.max())
        p = ex / ex.sum()
        wts = p[order]
        if c.renormalize:
            wts = wts / wts.sum()
        for e, wt in zip(order, wts):
            w1 = ((c.fc1[e].astype(np.float32) - 128) *
                  _value(c.fc1_scales[e], dtype).astype(np.float32)[:, None]).astype(np.float64)
            w2 = ((c.fc2[e].astype(np.float32) - 128) *
                  _value(c.fc2_scales[e], dtype).astype(np.float32)[:, None]).astype(np.float64)
            x1 = w1 @ A[t]
            g, u = x1[:I], x1[I:]
            h = g / (1.0 + np.exp(-g)) * u
            h = h.astype(np.float16).astype(np.float64)
            out[si] += wt * (w2 @ h)
    return out


@pytest.mark.parametrize("renorm", [False, True])
def test_moe_brute_force(renorm):
    c = inputs.make_moe_case(T=6, H=64, I=32, E=5, topk=2, act_dtype=F16, case=1,
                             renormalize=renorm, config=9)
    got = oracle.moe_ffn(c.A, F16, c.logits, c.fc1, c.fc1_scales, c.fc2, c.fc2_scales,
                         c.T, c.H, c.I, c.E, c.topk, renormalize=renorm)
    ref = _brute_force_moe(c, list(range(c.T)), F16)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-12 * np.abs(ref).max())


def test_moe_token_subset_equals_full_rows():
    c = inputs.make_moe_case(T=9, H=64, I=32, E=4, topk=2, act_dtype=BF16, case=2, config=9)
    full = oracle.moe_ffn(c.A, BF16, c.logits, c.fc1, c.fc1_scales, c.fc2, c.fc2_scales,
                          c.T, c.H, c.I, c.E, c.topk, nthreads=3)
    sub = oracle.moe_ffn(c.A, BF16, c.logits, c.fc1, c.fc1_scales, c.fc2, c.fc2_scales,
                         c.T, c.H, c.I, c.E, c.topk, tokens=[7, 0, 4], nthreads=1)
    assert np.array_equal(sub, full[[7, 0, 4]])


def test_moe_neutral_fc2_gives_zero():
    c = inputs.make_moe_case(T=4, H=32, I=16, E=3, topk=2, act_dtype=BF16, case=3, config=9)
    c.fc2[:] = 128
    out = oracle.moe_ffn(c.A, BF16, c.logits, c.fc1, c.fc1_scales, c.fc2, c.fc2_scales,
                         c.T, c.H, c.I, c.E, c.topk)
    assert np.all(out == 0.0)


def test_moe_single_expert_is_two_gemms():
    # E = 1, top-1: out = fc2(round(silu(g) * u)) with weight softmax = 1
    c = inputs.make_moe_case(T=3, H=64, I=32, E=1, topk=1, act_dtype=F16, case=4, config=9)
    out = oracle.moe_ffn(c.A, F16, c.logits, c.fc1, c.fc1_scales, c.fc2, c.fc2_scales,
                         c.T, c.H, c.I, c.E, c.topk)
    x1 = oracle.gemm(c.A, F16, c.fc1[0], c.fc1_scales[0], None, None, 3, 64, 64, -1, 8)
    g, u = x1[:, :32], x1[:, 32:]
    h = (g / (1.0 + np.exp(-g)) * u).astype(np.float16).view(np.uint16)
    y = oracle.gemm(h, F16, c.fc2[0], c.fc2_scales[0], None, None, 3, 64, 32, -1, 8)
    assert np.allclose(out, y, rtol=1e-13, atol=1e-15)
    assert math.isfinite(float(out.sum()))
