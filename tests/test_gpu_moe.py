"""GPU parity of wo_moe_ffn (routing, grouped fc1 with the gated activation,
grouped fc2, weighted combine) against the oracle's MoE FFN on the same
seeded inputs: every output at small sizes, sampled tokens at the full
workload size (T=1024, 64 experts, top-2, hidden 4096, inter 1408)."""
import numpy as np
import pytest

import oracle
from helpers import assert_within_tolerance, from_device_bits, to_device_bits, to_device_u8
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


class DeviceMoe:
    def __init__(self, wo, c):
        self.c = c
        self.A = to_device_bits(c.A, c.act_dtype)
        self.logits = torch.from_numpy(c.logits).cuda()
        self.fc1 = wo.pack_experts(to_device_u8(c.fc1), c.E, 2 * c.I, c.H, 8)
        self.fc2 = wo.pack_experts(to_device_u8(c.fc2), c.E, c.H, c.I, 8)
        self.s1 = to_device_bits(c.fc1_scales, c.act_dtype)
        self.s2 = to_device_bits(c.fc2_scales, c.act_dtype)
        self.wo = wo

    def run(self, workspace=None):
        c = self.c
        return self.wo.moe_ffn(self.A, self.logits, self.fc1, self.s1, self.fc2, self.s2, c.H,
                               c.I, c.E, c.topk, renormalize=c.renormalize,
                               workspace=workspace)

    def oracle(self, tokens=None):
        c = self.c
        return oracle.moe_ffn(c.A, c.act_dtype, c.logits, c.fc1, c.fc1_scales, c.fc2,
                              c.fc2_scales, c.T, c.H, c.I, c.E, c.topk,
                              renormalize=c.renormalize, tokens=tokens)


@pytest.mark.parametrize("T,H,I,E,topk,act,renorm", [
    (37, 256, 128, 8, 2, inputs.BF16, False),
    (64, 512, 192, 16, 2, inputs.F16, True),
    (5, 128, 64, 4, 1, inputs.BF16, False),
    (300, 256, 256, 6, 3, inputs.BF16, False),   # > 64 rows per expert: several passes
    (48, 384, 128, 12, 4, inputs.F16, True),     # tensor-core experts, fp16, top-4
    (6, 256, 128, 32, 2, inputs.BF16, False),    # most experts without rows
])
def test_moe_small(wo, T, H, I, E, topk, act, renorm):
    c = inputs.make_moe_case(T=T, H=H, I=I, E=E, topk=topk, act_dtype=act, case=T + E,
                             renormalize=renorm, config=9)
    dm = DeviceMoe(wo, c)
    out = dm.run()
    torch.cuda.synchronize()
    assert_within_tolerance(from_device_bits(out), act, dm.oracle(), f"moe T{T} E{E}")


def test_moe_routing_ties_pick_lower_expert(wo):
    c = inputs.make_moe_case(T=16, H=128, I=64, E=8, topk=2, act_dtype=inputs.BF16, case=5,
                             config=9)
    c.logits[:] = 0.0
    c.logits[:, 3] = 1.0           # one clear winner, then a seven-way tie at 0
    c.logits[5, :] = 2.0           # an all-way tie
    dm = DeviceMoe(wo, c)
    out = dm.run()
    torch.cuda.synchronize()
    assert_within_tolerance(from_device_bits(out), inputs.BF16, dm.oracle(), "ties")


def test_moe_full_size_sampled_tokens(wo):
    c = inputs.make_moe_case()     # T=1024, H=4096, I=1408, E=64, top-2, bf16
    dm = DeviceMoe(wo, c)
    out = dm.run()
    torch.cuda.synchronize()
    # 64 tokens: the first and last, and random ones in between
    rng = np.random.default_rng(5)
    tokens = np.unique(np.concatenate([[0, c.T - 1], rng.choice(np.arange(1, c.T - 1), 62,
                                                                 replace=False)]))
    got = from_device_bits(out)[tokens]
    assert_within_tolerance(got, inputs.BF16, dm.oracle(tokens), "moe full size")


def test_moe_deterministic(wo):
    c = inputs.make_moe_case(T=256, H=512, I=256, E=16, topk=2, case=7, config=9)
    dm = DeviceMoe(wo, c)
    a = dm.run().clone()
    b = dm.run().clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_moe_rejects_bad_arguments(wo):
    c = inputs.make_moe_case(T=4, H=128, I=64, E=4, topk=2, case=8, config=9)
    dm = DeviceMoe(wo, c)
    with pytest.raises(wo.WoError):
        wo.moe_ffn(dm.A, dm.logits, dm.fc1, dm.s1, dm.fc2, dm.s2, 100, 64, 4, 2)
    with pytest.raises(wo.WoError):
        wo.moe_ffn(dm.A, dm.logits, dm.fc1, dm.s1, dm.fc2, dm.s2, 128, 64, 4, 5)
