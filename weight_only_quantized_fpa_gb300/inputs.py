"""Seeded synthetic inputs for the weight-only GEMM workloads.

This module only draws random numbers and stores them in the dtypes the
operation takes (fp16/bf16 bit patterns as uint16, uint8 codes, fp32 logits).
It holds none of the operation's arithmetic, so both the CUDA path and the CPU
oracle can be fed from it.

Recipe (one numpy PCG64 stream per tensor, seed = 0x5EED0000 + 4096*config +
16*case + tensor id):

* A (activations): standard normal drawn in fp64, rounded to nearest even
  into fp16 or bf16;
* int8 codes: uniform bytes 0..255; int4 codes: uniform bytes 0..255, i.e. two
  independent uniform nibbles per byte, which is the row-major packed form
  (byte j = code 2j | code 2j+1 << 4) of uniform 0..15 codes;
* scales: uniform on [lo, hi) in fp64, rounded into the activation dtype;
* zeros: normal with standard deviation 0.01; bias: normal with standard
  deviation 0.1 (the second parameter of N(mu, sigma) read as sigma);
* gating logits: standard normal, fp32;
* act-order group index (GPTQ ``g_idx``): a uniformly random order of the k
  input channels stands in for the quantiser's column order; the i-th
  channel in that order belongs to group i // group_size, so every group has
  group_size channels scattered over k.

Tensor ids: A=1, codes=2, scale=3, zero=4, bias=5, logits=6, fc1 codes=7,
fc1 scales=8, fc2 codes=9, fc2 scales=10, g_idx=11.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F16 = 0
BF16 = 1

T_A, T_CODES, T_SCALE, T_ZERO, T_BIAS, T_LOGITS = 1, 2, 3, 4, 5, 6
T_FC1, T_FC1_S, T_FC2, T_FC2_S = 7, 8, 9, 10
T_GIDX = 11


def seed_for(config: int, case: int, tensor: int) -> int:
    return 0x5EED0000 + 4096 * config + 16 * case + tensor


def rng_for(config: int, case: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_for(config, case, tensor)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """fp64/fp32 values -> fp16 or bf16 bit patterns (round to nearest even)."""
    if dtype == F16:
        return np.ascontiguousarray(x).astype(np.float16).view(np.uint16)
    # bf16: the fp64 draw is rounded to fp32 and then to bf16 (both to nearest
    # even).  The stored bits are the input; both sides read the same bits.
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def normal_bits(rng, shape, dtype, sigma=1.0) -> np.ndarray:
    return to_bits(rng.standard_normal(shape) * sigma, dtype)


def uniform_bits(rng, shape, dtype, lo, hi) -> np.ndarray:
    return to_bits(rng.uniform(lo, hi, shape), dtype)


def code_bytes(rng, shape) -> np.ndarray:
    return rng.integers(0, 256, size=shape, dtype=np.uint8)


def act_order_g_idx(rng, k: int, group_size: int) -> np.ndarray:
    """int32 [k] group index of an act-order checkpoint (see the recipe)."""
    order = rng.permutation(k)
    g = np.empty(k, dtype=np.int32)
    g[order] = np.arange(k, dtype=np.int32) // group_size
    return g


@dataclass
class GemmCase:
    """One weight-only GEMM problem, host-side arrays."""
    name: str
    m: int
    n: int
    k: int
    bits: int
    group_size: int
    act_dtype: int
    A: np.ndarray            # uint16 [m, k]
    B: np.ndarray            # uint8 [n, k] (bits 8) or [n, k/2] (bits 4), row-major
    scales: np.ndarray       # uint16 [n] or [n, k/group]
    zeros: np.ndarray | None
    bias: np.ndarray | None
    g_idx: np.ndarray | None = None  # int32 [k]: act-order group of each input channel

    @property
    def weight_bytes(self) -> int:
        b = self.B.nbytes + self.scales.nbytes
        if self.zeros is not None:
            b += self.zeros.nbytes
        return b


def make_gemm_case(config: int, case: int, m: int, n: int, k: int, *, bits: int,
                   group_size: int, act_dtype: int, scale_lo: float, scale_hi: float,
                   with_zeros: bool, with_bias: bool, name: str = "",
                   act_order: bool = False) -> GemmCase:
    A = normal_bits(rng_for(config, case, T_A), (m, k), act_dtype)
    if bits == 8:
        B = code_bytes(rng_for(config, case, T_CODES), (n, k))
    else:
        B = code_bytes(rng_for(config, case, T_CODES), (n, k // 2))
    per_channel = group_size in (-1, k)
    sshape = (n,) if per_channel else (n, k // group_size)
    scales = uniform_bits(rng_for(config, case, T_SCALE), sshape, act_dtype,
                          scale_lo, scale_hi)
    zeros = (normal_bits(rng_for(config, case, T_ZERO), sshape, act_dtype, 0.01)
             if with_zeros else None)
    bias = (normal_bits(rng_for(config, case, T_BIAS), (n,), act_dtype, 0.1)
            if with_bias else None)
    g_idx = (act_order_g_idx(rng_for(config, case, T_GIDX), k, k if per_channel else group_size)
             if act_order else None)
    return GemmCase(name or f"cfg{config}.case{case}", m, n, k, bits, group_size,
                    act_dtype, A, B, scales, zeros, bias, g_idx)


# -- the five workloads ------------------------------------------------------

W4_TINY = dict(config=1, shapes=[(1, 256, 512)], bits=4, group_size=64, act_dtype=BF16,
               scale_lo=0.005, scale_hi=0.02, with_zeros=True, with_bias=False)

W8_DECODE_NK = [(4608, 3584), (3584, 3584), (37888, 3584), (3584, 18944)]
W8_DECODE = dict(config=2, shapes=[(m, n, k) for m in (1, 4, 16) for (n, k) in W8_DECODE_NK],
                 bits=8, group_size=-1, act_dtype=F16, scale_lo=0.001, scale_hi=0.01,
                 with_zeros=False, with_bias=True)

W8_LARGE_NK = [(2048, 2048), (4096, 4096), (4608, 3584)]
W8_LARGE = dict(config=3, shapes=[(m, n, k) for m in (256, 1024, 4096, 8192)
                                  for (n, k) in W8_LARGE_NK],
                bits=8, group_size=-1, act_dtype=F16, scale_lo=0.001, scale_hi=0.01,
                with_zeros=False, with_bias=False)

W4_G64_NK = [(2048, 2048), (3072, 2048), (13312, 2048), (131072, 2048), (2048, 13312)]
W4_G64 = dict(config=4, shapes=[(m, n, k) for m in (1, 512) for (n, k) in W4_G64_NK],
              bits=4, group_size=64, act_dtype=BF16, scale_lo=0.005, scale_hi=0.02,
              with_zeros=True, with_bias=False)

# GPTQ act-order (g_idx), group 128, on the shapes of the group-64 workload
W4_ACT_ORDER = dict(config=6, shapes=[(m, n, k) for m in (1, 512) for (n, k) in W4_G64_NK],
                    bits=4, group_size=128, act_dtype=BF16, scale_lo=0.005, scale_hi=0.02,
                    with_zeros=True, with_bias=False, act_order=True)

# the same without act-order (channels in order, group 128)
W4_G128 = dict(W4_ACT_ORDER, config=7, act_order=False)

# the other activation dtype with each code width (bf16 with 8-bit decode,
# fp16 with 4-bit), per-channel 4-bit, and 8-bit decode at 17..64 rows
W8_DECODE_BF16 = dict(W8_DECODE, config=8, act_dtype=BF16)
W4_G64_F16 = dict(W4_G64, config=9, act_dtype=F16)
W4_PER_CHANNEL = dict(W4_G64, config=10, group_size=-1)
W8_MID = dict(W8_DECODE, config=11, shapes=[(m, n, k) for m in (24, 32, 48, 64)
                                            for (n, k) in W8_DECODE_NK])

GEMM_WORKLOADS = {1: W4_TINY, 2: W8_DECODE, 3: W8_LARGE, 4: W4_G64, 6: W4_ACT_ORDER, 7: W4_G128,
                  8: W8_DECODE_BF16, 9: W4_G64_F16, 10: W4_PER_CHANNEL, 11: W8_MID}


def workload_case(config: int, case: int) -> GemmCase:
    """Case `case` (index into the workload's shape list) of GEMM workload `config`."""
    w = GEMM_WORKLOADS[config]
    m, n, k = w["shapes"][case]
    return make_gemm_case(config, case, m, n, k, bits=w["bits"], group_size=w["group_size"],
                          act_dtype=w["act_dtype"], scale_lo=w["scale_lo"],
                          scale_hi=w["scale_hi"], with_zeros=w["with_zeros"],
                          with_bias=w["with_bias"], name=f"cfg{config}:m{m}n{n}k{k}",
                          act_order=w.get("act_order", False))


@dataclass
class MoeCase:
    T: int
    H: int
    I: int
    E: int
    topk: int
    act_dtype: int
    A: np.ndarray           # uint16 [T, H]
    logits: np.ndarray      # float32 [T, E]
    fc1: np.ndarray         # uint8 [E, 2I, H]
    fc1_scales: np.ndarray  # uint16 [E, 2I]
    fc2: np.ndarray         # uint8 [E, H, I]
    fc2_scales: np.ndarray  # uint16 [E, H]
    renormalize: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def weight_bytes(self) -> int:
        return (self.fc1.nbytes + self.fc1_scales.nbytes + self.fc2.nbytes
                + self.fc2_scales.nbytes)


def make_moe_case(T=1024, H=4096, I=1408, E=64, topk=2, act_dtype=BF16, case=0,
                  renormalize=False, config=5) -> MoeCase:
    A = normal_bits(rng_for(config, case, T_A), (T, H), act_dtype)
    logits = rng_for(config, case, T_LOGITS).standard_normal((T, E)).astype(np.float32)
    fc1 = code_bytes(rng_for(config, case, T_FC1), (E, 2 * I, H))
    fc1_s = uniform_bits(rng_for(config, case, T_FC1_S), (E, 2 * I), act_dtype, 0.001, 0.01)
    fc2 = code_bytes(rng_for(config, case, T_FC2), (E, H, I))
    fc2_s = uniform_bits(rng_for(config, case, T_FC2_S), (E, H), act_dtype, 0.001, 0.01)
    return MoeCase(T, H, I, E, topk, act_dtype, A, logits, fc1, fc1_s, fc2, fc2_s,
                   renormalize)
