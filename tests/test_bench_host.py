"""CPU tests of bench.py's host logic: launch counting, the DRAM-traffic
lookup, and the workloads' case lists."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from weight_only_quantized_fpa_gb300 import inputs  # noqa: E402


def test_launch_count_per_call():
    c = inputs.make_gemm_case(9, 0, 1, 64, 128, bits=4, group_size=64, act_dtype=inputs.BF16,
                              scale_lo=0.01, scale_hi=0.02, with_zeros=True, with_bias=False)
    assert bench.case_launches(c) == 1                       # streaming kernel
    c.m = 512
    assert bench.case_launches(c) == 2                       # 4-bit prepass + tensor cores
    c.act_dtype = inputs.F16
    assert bench.case_launches(c) == 2                       # the prepass runs for fp16 A too
    c.bits = 8
    assert bench.case_launches(c) == 1                       # 8-bit: the GEMM kernel alone
    c.bits = 4
    c.g_idx = np.zeros(c.k, dtype=np.int32)
    assert bench.case_launches(c) == 3                       # + the act-order gather
    c.m = 1
    assert bench.case_launches(c) == 2


def test_traffic_is_reported_only_for_its_workload_and_source():
    src = ["wo_stream.cu", "wo_common.cuh", "wo_sm100.cuh"]
    h = bench.kernel_source_hash(src)
    e = bench.traffic_from_profile("stream_kernel", h, "w8_decode")
    if e is None:
        pytest.skip("stream_kernel changed since its DRAM traffic was captured")
    assert e["bench_workload"] == "w8_decode"
    assert bench.traffic_from_profile("stream_kernel", h, "w4_g64") is None
    assert bench.traffic_from_profile("stream_kernel", "0" * 16, "w8_decode") is None


@pytest.mark.parametrize("name", ["w4_act_order", "w4_g128"])
def test_group128_workloads_share_shapes(name):
    cases = bench.workload_cases(name)
    assert [(c.m, c.n, c.k) for c in cases] == inputs.W4_G64["shapes"]
    for c in cases[:3]:
        assert c.group_size == 128 and c.bits == 4
        if name == "w4_act_order":
            # every group holds exactly 128 channels
            assert np.array_equal(np.bincount(c.g_idx), np.full(c.k // 128, 128))
        else:
            assert c.g_idx is None


def test_reference_arm_prints_one_contract_line():
    # the reference arm runs the oracle on the host cores: one JSON line with
    # the contract's keys
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "w4_tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ["impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"]:
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


@pytest.mark.parametrize("n,k", [(2048, 2048), (131072, 2048), (2048, 13312)])
def test_w4_g64_bytes_are_four_and_a_half_bits_per_weight(n, k):
    # vLLM-Omni "cpu_int4.py", module docstring: 4-bit codes with a bf16 scale
    # and offset per group of 64 are 4.5 bits per weight.  The bench's
    # algorithmic bytes (the roofline's numerator) must count exactly that.
    c = inputs.make_gemm_case(4, 0, 1, n, k, bits=4, group_size=64, act_dtype=inputs.BF16,
                              scale_lo=0.005, scale_hi=0.02, with_zeros=True, with_bias=False)
    assert c.weight_bytes * 8 == 4.5 * n * k


def test_w8_per_channel_bytes_are_codes_plus_one_scale_per_channel():
    # "acext User Guide (v1.7)" 1.3.1: one int8 per weight and a single scale
    # per output channel
    n, k = 4608, 3584
    c = inputs.make_gemm_case(2, 0, 1, n, k, bits=8, group_size=-1, act_dtype=inputs.F16,
                              scale_lo=0.001, scale_hi=0.01, with_zeros=False, with_bias=True)
    assert c.weight_bytes == n * k + 2 * n


@pytest.mark.parametrize("name,act,group,ms", [
    ("w8_decode_bf16", inputs.BF16, -1, {1, 4, 16}),
    ("w4_g64_f16", inputs.F16, 64, {1, 512}),
    ("w4_per_channel", inputs.BF16, -1, {1, 512}),
    ("w8_mid", inputs.F16, -1, {24, 32, 48, 64})])
def test_widened_workloads(name, act, group, ms):
    w = bench.WORKLOADS[name]
    cfg = inputs.GEMM_WORKLOADS[w["config"]]
    assert cfg["act_dtype"] == act and cfg["group_size"] == group
    assert {m for (m, _, _) in cfg["shapes"]} == ms
    assert w["dtype"] == ("bf16" if act == inputs.BF16 else "f16")
    c = inputs.workload_case(w["config"], 0)
    assert c.act_dtype == act and c.scales.shape == ((c.n,) if group == -1 else (c.n, c.k // group))


@pytest.mark.parametrize("name,kernel", [("w8_decode", "stream_kernel"), ("w8_large", "gemm_tc_kernel"),
                                         ("w8_mid", "gemm_tc_kernel")])
def test_roofline_kernel_follows_the_plans(name, kernel):
    # the roofline names the kernel that carries most of the step's bytes (or
    # flops) by the library's own plan of each case; w8_mid's bytes are mostly
    # the 37888-channel cases, which have more 128-channel blocks than SMs and
    # so run on the tensor-core kernel
    import weight_only_quantized_fpa_gb300 as wo
    wo.load_library()
    k, src = bench.dominant_kernel(wo, bench.workload_cases(name), bench.WORKLOADS[name]["unit"] != "GB/s")
    assert k == kernel and all(os.path.exists(os.path.join(ROOT, "weight_only_quantized_fpa_gb300", "csrc", f))
                               for f in src)
