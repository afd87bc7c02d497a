"""GPU parity of wo_embed (rows of a packed quantised vocab table,
dequantised; vLLM-Omni "cpu_int4.py" CPUInt4EmbeddingMethod.embedding)
against the oracle: bit-identical, since both round the same fp32 value
once."""
import numpy as np
import pytest

import oracle
from helpers import DeviceCase, from_device_bits
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


def _ids(vocab, T, seed):
    rng = np.random.default_rng(seed)
    edge = [0, 1, 7, 8, 15, 16, 17, vocab - 17, vocab - 16, vocab - 1, -1, vocab, -5, vocab + 100]
    return np.concatenate([np.array(edge, dtype=np.int32),
                           rng.integers(0, vocab, size=T, dtype=np.int32)])


def _check(wo, c, ids):
    dc = DeviceCase(c)
    ids_d = torch.from_numpy(ids).cuda()
    out = wo.embed(ids_d, dc.B, dc.scales, c.n, c.k, c.bits, group_size=c.group_size,
                   zeros=dc.zeros)
    torch.cuda.synchronize()
    ref = oracle.embed(ids, c.B, c.scales, c.zeros, c.n, c.k, c.group_size, c.bits, c.act_dtype)
    got = from_device_bits(out)
    assert got.shape == ref.shape
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:4].tolist()}"


@pytest.mark.parametrize("vocab,hidden,bits,group,act,zeros", [
    (256, 512, 8, -1, inputs.F16, False),
    (192, 1024, 8, -1, inputs.BF16, False),
    (320, 1024, 4, 64, inputs.BF16, True),
    (128, 768, 4, 128, inputs.F16, True),
    (64, 512, 4, -1, inputs.BF16, True),   # per-channel 4-bit
    (128, 256, 4, 64, inputs.F16, False),  # no zeros
])
def test_embed_small(wo, vocab, hidden, bits, group, act, zeros):
    c = inputs.make_gemm_case(11, vocab + hidden + bits, 1, vocab, hidden, bits=bits,
                              group_size=group, act_dtype=act,
                              scale_lo=0.005 if bits == 4 else 0.001,
                              scale_hi=0.02 if bits == 4 else 0.01, with_zeros=zeros,
                              with_bias=False)
    _check(wo, c, _ids(vocab, 50, vocab + hidden))


def test_embed_vocab_table(wo):
    # the W4 group-64 workload's 131072 x 2048 head, read as a vocab table
    c = inputs.workload_case(4, 3)
    assert (c.n, c.k) == (131072, 2048)
    _check(wo, c, _ids(c.n, 200, 7))


def test_embed_empty_is_noop(wo):
    c = inputs.make_gemm_case(11, 1, 1, 64, 128, bits=4, group_size=64, act_dtype=inputs.BF16,
                              scale_lo=0.005, scale_hi=0.02, with_zeros=True, with_bias=False)
    dc = DeviceCase(c)
    out = wo.embed(torch.empty(0, dtype=torch.int32, device="cuda"), dc.B, dc.scales, 64, 128, 4,
                   group_size=64, zeros=dc.zeros)
    assert out.shape == (0, 128)
