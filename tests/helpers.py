"""Shared helpers for the parity tests (not collected as tests)."""
from __future__ import annotations

import numpy as np

import oracle
from weight_only_quantized_fpa_gb300 import inputs

# Tolerances of the weight-only GEMM against the fp64 oracle, on all m x n
# outputs (or on the sampled rows at full size).
REL_L2_TOL = 2e-3
MAX_ABS_TOL = 1e-2  # times max |C_ref|


def torch_dtype(act: int):
    import torch
    return torch.float16 if act == inputs.F16 else torch.bfloat16


def to_device_bits(arr_u16: np.ndarray, act: int, device="cuda"):
    """uint16 bit patterns -> a torch fp16/bf16 tensor on the device."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(arr_u16).view(np.int16))
    return t.to(device).view(torch_dtype(act))


def to_device_u8(arr: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def from_device_bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def error_stats(C_bits: np.ndarray, act: int, C_ref: np.ndarray):
    got = oracle.decode(C_bits, act)
    diff = got - C_ref
    rel_l2 = float(np.linalg.norm(diff) / max(np.linalg.norm(C_ref), 1e-300))
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    ref_max = float(np.abs(C_ref).max()) if C_ref.size else 0.0
    floor = oracle.decode(oracle.round_to(C_ref, act), act) - C_ref
    floor_l2 = float(np.linalg.norm(floor) / max(np.linalg.norm(C_ref), 1e-300))
    return dict(rel_l2=rel_l2, max_abs=max_abs, ref_max=ref_max, floor_rel_l2=floor_l2,
                finite=bool(np.isfinite(got).all()))


def assert_within_tolerance(C_bits, act, C_ref, what=""):
    st = error_stats(C_bits, act, C_ref)
    assert st["finite"], f"{what}: non-finite output"
    assert st["rel_l2"] <= REL_L2_TOL, f"{what}: rel_L2 {st['rel_l2']:.3e} (floor {st['floor_rel_l2']:.3e})"
    assert st["max_abs"] <= MAX_ABS_TOL * st["ref_max"] + 1e-30, \
        f"{what}: max|dC| {st['max_abs']:.3e} vs max|C| {st['ref_max']:.3e}"
    return st


class DeviceCase:
    """A GemmCase uploaded to the GPU and packed with wo_pack."""

    def __init__(self, case: inputs.GemmCase, device="cuda"):
        import weight_only_quantized_fpa_gb300 as wo
        self.c = case
        self.A = to_device_bits(case.A, case.act_dtype, device)
        self.B_rowmajor = to_device_u8(case.B, device)
        self.B = wo.pack(self.B_rowmajor, case.n, case.k, case.bits)
        self.scales = to_device_bits(case.scales, case.act_dtype, device)
        self.zeros = None if case.zeros is None else to_device_bits(case.zeros, case.act_dtype, device)
        self.bias = None if case.bias is None else to_device_bits(case.bias, case.act_dtype, device)

    def run(self, A=None, out=None, workspace=None):
        import weight_only_quantized_fpa_gb300 as wo
        c = self.c
        return wo.gemm(self.A if A is None else A, self.B, self.scales, c.n, c.k, c.bits,
                       group_size=c.group_size, zeros=self.zeros, bias=self.bias, out=out,
                       workspace=workspace)

    def oracle_rows(self, rows=None) -> np.ndarray:
        c = self.c
        A = c.A if rows is None else c.A[rows]
        m = A.shape[0]
        return oracle.gemm(A, c.act_dtype, c.B, c.scales, c.zeros, c.bias, m, c.n, c.k,
                           c.group_size, c.bits)


def sample_rows(m: int, count: int = 64, seed: int = 0) -> np.ndarray:
    """At least `count` rows (all rows when m <= count), sorted and unique: the
    first and last row, one row in every 128-row block (so both 128-row halves
    of a 256-row tile, every tile a persistent CTA runs as its second or later
    unit, and the ragged last tile are all checked; the row within the block
    moves through the four 32-row TMEM lane quadrants from block to block),
    then random rows up to `count`."""
    if m <= count:
        return np.arange(m)
    rng = np.random.default_rng(seed)
    rows = {0, m - 1}
    for b, b0 in enumerate(range(0, m, 128)):
        rows.add(min(b0 + 32 * (b % 4) + int(rng.integers(0, 32)), m - 1))
    free = np.setdiff1d(np.arange(m), np.fromiter(rows, dtype=np.int64))
    need = count - len(rows)
    if need > 0:
        rows.update(rng.choice(free, size=need, replace=False).tolist())
    return np.array(sorted(rows))
