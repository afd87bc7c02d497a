#!/usr/bin/env python
"""Benchmark of the weight-only quantized GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload w8_decode|w4_g64|w8_large|w4_tiny|moe]

One step is one pass of the hot path over the workload's batch: one wo_gemm
per (m, N, K) case of the workload, each case with its own weights.  The
default workload is the A16W8 per-channel decode set (fp16 A with m in
{1, 4, 16}, uint8 codes, fp16 scale and bias; (N, K) in {(4608,3584),
(3584,3584), (37888,3584), (3584,18944)}), reported as effective weight GB/s
(packed code bytes + scale bytes per second).

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and torch.cuda.synchronize(); a step is one CUDA graph holding every case's
kernel back to back, timed with CUDA events on the launching stream.  The 12
decode cases read 12 distinct weight matrices (about 700 MB per step, over
five times the L2), so every launch streams its weights from HBM.  A
per-case breakdown is measured afterwards, each case replayed alone between
the others.

Rank 0 prints one JSON line.  `--impl reference` times the CPU oracle (the
plain C implementation the tests check against) on a bounded sample of the
same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from weight_only_quantized_fpa_gb300 import inputs  # noqa: E402

METRIC = "weight-only GEMM: weight GB/s (m≤16), TFLOP/s (m≥64), % of roofline"

WORKLOADS = {
    "w8_decode": dict(config=2, unit="GB/s", dtype="f16",
                      desc="A16W8 per-channel decode: fp16 A [m,K] ~N(0,1), m in {1,4,16}; "
                           "uint8 codes w=(q-128)*s, fp16 scale [N] ~U(0.001,0.01), fp16 bias "
                           "~N(0,0.1); (N,K) in {(4608,3584),(3584,3584),(37888,3584),"
                           "(3584,18944)}"),
    "w4_g64": dict(config=4, unit="GB/s", dtype="bf16",
                   desc="W4A16 group-64 asymmetric, bf16: m in {1,512}; (N,K) in "
                        "{(2048,2048),(3072,2048),(13312,2048),(131072,2048),(2048,13312)}"),
    "w8_large": dict(config=3, unit="TFLOP/s", dtype="f16",
                     desc="A16W8 per-channel large m: m in {256,1024,4096,8192}; (N,K) in "
                          "{(2048,2048),(4096,4096),(4608,3584)}, fp16"),
    "w4_act_order": dict(config=6, unit="GB/s", dtype="bf16",
                         desc="W4A16 GPTQ act-order (g_idx), group 128, asymmetric, bf16: the "
                              "w4_g64 shapes (m in {1,512}; (N,K) in {(2048,2048),(3072,2048),"
                              "(13312,2048),(131072,2048),(2048,13312)}); g_idx = a random "
                              "channel order cut into groups of 128; bytes = codes, scales, "
                              "zeros"),
    "w4_g128": dict(config=7, unit="GB/s", dtype="bf16",
                    desc="W4A16 group 128, asymmetric, bf16, channels in order: the w4_act_order "
                         "shapes and value distributions without the act-order group index"),
    "w8_decode_bf16": dict(config=8, unit="GB/s", dtype="bf16",
                           desc="A16W8 per-channel decode with bf16 activations, scales and "
                                "bias: the w8_decode shapes (m in {1,4,16})"),
    "w4_g64_f16": dict(config=9, unit="GB/s", dtype="f16",
                       desc="W4A16 group 64 with fp16 activations, scales and zeros: the w4_g64 "
                            "shapes (m in {1,512})"),
    "w4_per_channel": dict(config=10, unit="GB/s", dtype="bf16",
                           desc="4-bit codes with one bf16 scale and zero per output channel: "
                                "the w4_g64 shapes (m in {1,512})"),
    "w8_mid": dict(config=11, unit="GB/s", dtype="f16",
                   desc="A16W8 per-channel, fp16, m in {24,32,48,64} (between decode and the "
                        "tensor-core sizes) on the w8_decode (N,K)"),
    "w4_tiny": dict(config=1, unit="GB/s", dtype="bf16",
                    desc="W4A16 tiny: m=1, N=256, K=512, group 64, bf16"),
    "moe": dict(config=5, unit="GB/s", dtype="bf16",
                desc="MoE grouped weight-only FFN: T=1024 tokens, 64 experts, top-2 of softmax "
                     "of fp32 logits ~N(0,1); hidden 4096, inter 1408; per expert fc1 "
                     "[2816,4096] and fc2 [4096,1408] int8 per-channel, bf16 scales "
                     "~U(0.001,0.01); SiLU-gated fc1, fc2, routing-weighted sum; A bf16 ~N(0,1)"),
    "embed": dict(config=4, unit="GB/s", dtype="bf16",
                  desc="Packed-embedding row gather (wo_embed): 16384 token ids ~U[0,131072) per "
                       "call, 4 id sets rotated so the gathered rows exceed L2 across calls; the "
                       "table is the w4_g64 head (131072 x 2048, 4-bit group 64, bf16 scales and "
                       "zeros); bytes = the rows' codes, scales and zeros + the bf16 output"),
}
EMBED_T, EMBED_SETS = 16384, 4

HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="w8_decode")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing leg (for quick local runs)")
    ap.add_argument("--no-sub-records", action="store_true",
                    help="skip the large-m and steady-state sub-records of the default run")
    ap.add_argument("--profile-case", type=int, default=None, metavar="I",
                    help="profiling mode: run only case I of the workload, --steps calls, "
                         "and print no JSON (for ncu captures)")
    return ap.parse_args()


def run_profile_case(args):
    import torch

    import weight_only_quantized_fpa_gb300 as wo

    wo.load_library()
    c = workload_cases(args.workload)[args.profile_case]
    dt = torch.float16 if c.act_dtype == inputs.F16 else torch.bfloat16

    def up16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(dt)

    A, s = up16(c.A), up16(c.scales)
    z = None if c.zeros is None else up16(c.zeros)
    b = None if c.bias is None else up16(c.bias)
    if c.g_idx is not None:  # act-order: group-sorted pack, gather per call
        perm = wo.act_order_perm(c.g_idx, c.k, c.group_size).cuda()
        B = wo.pack_act_order(torch.from_numpy(c.B).cuda(), perm, c.n, c.k, c.bits)
        for _ in range(args.steps):
            wo.gemm_act_order(A, B, perm, s, c.n, c.k, c.bits, c.group_size, zeros=z, bias=b)
        torch.cuda.synchronize()
        print(f"profiled {c.name}: {args.steps} calls", file=sys.stderr)
        return 0
    B = wo.pack(torch.from_numpy(c.B).cuda(), c.n, c.k, c.bits)
    for _ in range(args.steps):
        wo.gemm(A, B, s, c.n, c.k, c.bits, group_size=c.group_size, zeros=z, bias=b)
    torch.cuda.synchronize()
    print(f"profiled {c.name}: {args.steps} calls", file=sys.stderr)
    return 0


# ------------------------------------------------------------- workload ---

def workload_cases(name: str):
    w = WORKLOADS[name]
    cfg = inputs.GEMM_WORKLOADS[w["config"]]
    return [inputs.workload_case(w["config"], i) for i in range(len(cfg["shapes"]))]


def case_flops(c) -> float:
    return 2.0 * c.m * c.n * c.k


def case_launches(c) -> int:
    """This library's kernels per GEMM call: the act-order column gather, the
    4-bit prepass of the tensor-core kernel (channel scales into fp16 range,
    bf16 activations into fp16), the GEMM kernel."""
    tc = c.m >= 65
    return (c.g_idx is not None) + (tc and c.bits == 4) + 1


# wo_gemm_plan's kernel -> the CUDA kernel that runs it and its sources
PLAN_KERNELS = {
    "stream": ("stream_kernel", ["wo_stream.cu", "wo_common.cuh", "wo_sm100.cuh"]),
    "stream_persistent": ("gemv4_kernel", ["wo_gemv.cu", "wo_common.cuh", "wo_sm100.cuh"]),
    "tensor_core": ("gemm_tc_kernel", ["wo_gemm_tc.cu", "wo_common.cuh", "wo_sm100.cuh"]),
    "tensor_core_swap_ab": ("moe_tc_kernel", ["wo_gemm_tc.cu", "wo_common.cuh", "wo_sm100.cuh"]),
}


def dominant_kernel(wo, cases, by_flops: bool):
    """The GEMM kernel that carries the largest share of a step's algorithmic
    bytes (or flops), by the library's own plan of each case: (name, sources)."""
    share = {}
    for c in cases:
        k = wo.gemm_plan(c.m, c.n, c.k, c.bits, c.group_size, c.act_dtype)["kernel"]
        share[k] = share.get(k, 0) + (case_flops(c) if by_flops else c.weight_bytes)
    return PLAN_KERNELS[max(share, key=share.get)]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, "fallback"


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "weight_only_quantized_fpa_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel: str, src_hash: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current kernel source and on this bench workload; else
    None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(kernel)
        if e and e.get("source_hash") == src_hash and e.get("bench_workload") == workload:
            return e
    except (OSError, ValueError):
        pass
    return None


# ---------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------- CPU baseline ----

def slice_case(c, n_sub: int):
    """The first n_sub output channels of a case (a bounded oracle sample)."""
    import copy
    s = copy.copy(c)
    s.n = n_sub
    s.B = c.B[:n_sub]
    s.scales = c.scales[:n_sub]
    s.zeros = None if c.zeros is None else c.zeros[:n_sub]
    s.bias = None if c.bias is None else c.bias[:n_sub]
    return s


def oracle_pass(cases, frac: float, threads: int):
    """Run the oracle over every case restricted to a fraction of its output
    channels (and of its rows for m > 64); returns (seconds, weight bytes,
    flops)."""
    import oracle
    t0 = time.perf_counter()
    wbytes = 0
    flops = 0.0
    for c in cases:
        n_sub = max(64, int(c.n * frac) // 64 * 64)
        s = slice_case(c, n_sub)
        m_sub = c.m if c.m <= 64 else max(1, int(c.m * frac))
        if s.g_idx is not None:
            oracle.gemm_gidx(s.A[:m_sub], s.act_dtype, s.B, s.scales, s.zeros, s.g_idx, s.bias,
                             m_sub, s.n, s.k, s.group_size, s.bits, nthreads=threads)
        else:
            oracle.gemm(s.A[:m_sub], s.act_dtype, s.B, s.scales, s.zeros, s.bias, m_sub, s.n,
                        s.k, s.group_size, s.bits, nthreads=threads)
        wbytes += s.weight_bytes
        flops += 2.0 * m_sub * s.n * s.k
    return time.perf_counter() - t0, wbytes, flops


def cpu_baseline(cases, unit, budget_s=10.0):
    threads = os.cpu_count() or 1
    frac = 1.0 / 64
    dt, wb, fl = oracle_pass(cases, frac, threads)
    # grow the sample toward the time budget (bounded: a few passes at most)
    if dt < budget_s / 4:
        frac = min(1.0, frac * max(1.0, budget_s / max(dt, 1e-3) / 2))
        dt, wb, fl = oracle_pass(cases, frac, threads)
    # a whole workload that takes well under the budget is repeated, so the
    # figure rests on about the budget's worth of CPU work
    reps = 1
    if frac >= 1.0 and dt < budget_s / 2:
        reps = max(1, min(100, int(budget_s / max(dt, 1e-3))))
        dt = wb = fl = 0.0
        for _ in range(reps):
            d, b, f = oracle_pass(cases, frac, threads)
            dt, wb, fl = dt + d, wb + b, fl + f
    value = wb / dt / 1e9 if unit == "GB/s" else fl / dt / 1e12
    return {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"every case of the workload on the first {frac:.4f} of its output "
                      f"channels (rows capped likewise above m=64), {reps} pass(es); "
                      f"{dt:.2f} s wall, {wb / 1e6:.1f} MB of weights"}


# ------------------------------------------------------------ distributed --

def dist_setup(backend: str | None = None):
    """Rank, world size and local rank from the torchrun environment; one
    process group for the barriers and the max over ranks (NCCL on GPUs,
    gloo where there are none, e.g. the CPU tests of this path)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, x: float) -> float:
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- arms -----

def run_reference_moe(args):
    import oracle
    oracle.build()
    w = WORKLOADS["moe"]
    c = inputs.make_moe_case()
    threads = os.cpu_count() or 1
    per_expert = c.weight_bytes / c.E
    per_step_budget = max(0.5, min(10.0, 120.0 / max(1, args.steps + args.warmup)))

    def one(ntok, first):
        tokens = (np.arange(ntok) + first) % c.T
        t0 = time.perf_counter()
        oracle.moe_ffn(c.A, c.act_dtype, c.logits, c.fc1, c.fc1_scales, c.fc2, c.fc2_scales,
                       c.T, c.H, c.I, c.E, c.topk, tokens=tokens, nthreads=threads)
        dt = time.perf_counter() - t0
        ids, _ = oracle.moe_route(c.logits[tokens], c.topk)
        return dt, len(set(ids.reshape(-1).tolist())) * per_expert

    dt, _ = one(2, 0)
    ntok = max(1, min(c.T, int(2 * per_step_budget / max(dt, 1e-3))))
    for i in range(args.warmup):
        one(ntok, i * ntok)
    tot_t = tot_b = 0.0
    for i in range(args.steps):
        dt, b = one(ntok, (args.warmup + i) * ntok)
        tot_t += dt
        tot_b += b
    value = tot_b / tot_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w["desc"]},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {ntok} consecutive tokens; bytes = the weights "
                                   "of the experts they route to"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def embed_bytes_per_row(c) -> int:
    G = c.k // 64
    return c.k // 2 + 2 * G * 2 + c.k * 2  # codes, scales and zeros, bf16 output


def run_reference_embed(args):
    import oracle
    oracle.build()
    w = WORKLOADS["embed"]
    c = inputs.workload_case(4, 3)
    rng = np.random.default_rng(1234)
    per_step_budget = max(0.5, min(10.0, 120.0 / max(1, args.steps + args.warmup)))

    def one(nids):
        ids = rng.integers(0, c.n, size=nids, dtype=np.int32)
        t0 = time.perf_counter()
        oracle.embed(ids, c.B, c.scales, c.zeros, c.n, c.k, c.group_size, c.bits, c.act_dtype)
        return time.perf_counter() - t0

    dt = one(64)
    nids = max(64, min(EMBED_T, int(64 * per_step_budget / max(dt, 1e-4))))
    for _ in range(args.warmup):
        one(nids)
    tot = sum(one(nids) for _ in range(args.steps))
    value = nids * args.steps * embed_bytes_per_row(c) / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w["desc"]},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: {nids} random ids of the table"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def embed_traffic():
    try:
        sh = kernel_source_hash(["wo_pack.cu", "wo_common.cuh"])
    except OSError:
        return None
    tr = traffic_from_profile("embed_kernel", sh, "embed")
    return tr["dram_bytes_per_launch"] if tr else None


def run_embed(args, ws, rank, local):
    import torch

    import weight_only_quantized_fpa_gb300 as wo

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wo.load_library()
    w = WORKLOADS["embed"]
    c = inputs.workload_case(4, 3)
    dt = torch.bfloat16

    def up16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt)

    B = wo.pack(torch.from_numpy(c.B).to(dev), c.n, c.k, c.bits)
    s, z = up16(c.scales), up16(c.zeros)
    rng = np.random.default_rng(1234 + rank)
    ids_h = [rng.integers(0, c.n, size=EMBED_T, dtype=np.int32) for _ in range(EMBED_SETS)]
    ids_d = [torch.from_numpy(x).to(dev) for x in ids_h]
    out = torch.empty((EMBED_T, c.k), dtype=dt, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call(ids, o):
        wo.wo_embed(ids, EMBED_T, B, s, z, o, c.n, c.k, c.group_size, c.bits, inputs.BF16, stream)

    with torch.cuda.stream(stream):
        call(ids_d[0], out)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()  # one replay = one call per id set
        with torch.cuda.graph(g, stream=stream):
            for i in range(EMBED_SETS):
                call(ids_d[i], out)
    torch.cuda.synchronize()
    bytes_per_call = EMBED_T * embed_bytes_per_row(c)
    sampler = ClockSampler(local)
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(args.steps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop()
    total_ms = max_over_ranks(ws, start.elapsed_time(end))
    calls = args.steps * EMBED_SETS
    value = bytes_per_call * calls * ws / (total_ms / 1e3) / 1e9

    # end to end: every call copies its ids in from pinned host memory and its
    # rows out, serially on one stream
    hI = [torch.from_numpy(x).pin_memory() for x in ids_h]
    hO = torch.empty((EMBED_T, c.k), dtype=dt, pin_memory=True)
    dI = torch.empty(EMBED_T, dtype=torch.int32, device=dev)
    e2e_calls = max(1, min(calls, 40))

    def e2e_call(i):
        with torch.cuda.stream(stream):
            dI.copy_(hI[i % EMBED_SETS], non_blocking=True)
            wo.embed(dI, B, s, c.n, c.k, c.bits, group_size=c.group_size, zeros=z, out=out,
                     stream=stream)
            hO.copy_(out, non_blocking=True)
    for i in range(3):
        e2e_call(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_calls):
        e2e_call(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(ws, time.perf_counter() - t0)
    if rank != 0:
        return 0
    hbm_gbs, _, peak_src = measured_peaks()
    achieved = bytes_per_call / (total_ms / calls / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w["desc"], "calls_per_step": EMBED_SETS,
                   "bytes_per_call": bytes_per_call,
                   "l2": "the 4 id sets gather 344 MB of rows and output per step: larger than L2",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "peak_source": f"hbm_gbs ({peak_src})",
                     "traffic": embed_traffic(), "kernel": "embed_kernel",
                     "algorithmic_bytes_per_launch": bytes_per_call,
                     "timing": f"{EMBED_SETS} launches per step in one CUDA graph"},
        "e2e": {"value": bytes_per_call * e2e_calls * ws / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": EMBED_T * 4, "d2h_bytes_per_step": EMBED_T * c.k * 2,
                "copies": "every call: pinned H2D of its ids, D2H of its rows, one stream"},
        "gpu_launches": calls,
        "clocks": clocks,
    }
    if ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        nids = 2048
        t0 = time.perf_counter()
        oracle.embed(ids_h[0][:nids], c.B, c.scales, c.zeros, c.n, c.k, c.group_size, c.bits,
                     c.act_dtype)
        dtc = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": nids * embed_bytes_per_row(c) / dtc / 1e9, "unit": "GB/s",
                                "cores": 1, "kind": "oracle",
                                "sample": f"{nids} of the ids, {dtc:.2f} s"}
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    if args.workload == "moe":
        return run_reference_moe(args)
    if args.workload == "embed":
        return run_reference_embed(args)
    w = WORKLOADS[args.workload]
    cases = workload_cases(args.workload)
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    # size one step so the whole run stays within about two minutes
    per_step_budget = max(0.2, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    frac = 1.0 / 256
    dt, _, _ = oracle_pass(cases, frac, threads)
    frac = max(1.0 / 1024, min(1.0, frac * per_step_budget / max(dt, 1e-3)))
    for _ in range(args.warmup):
        oracle_pass(cases, frac, threads)
    tot_t = tot_b = tot_f = 0.0
    for _ in range(args.steps):
        dt, wb, fl = oracle_pass(cases, frac, threads)
        tot_t += dt
        tot_b += wb
        tot_f += fl
    value = tot_b / tot_t / 1e9 if w["unit"] == "GB/s" else tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": w["unit"],
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": w["desc"], "cases": len(cases)},
        "cpu_baseline": {"value": value, "unit": w["unit"], "cores": threads, "kind": "oracle",
                         "sample": f"each step: every case on the first {frac:.5f} of its "
                                   "output channels (rows capped likewise above m=64)"},
        "e2e": {"value": value, "unit": w["unit"], "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_moe(args, ws, rank, local):
    import torch

    import weight_only_quantized_fpa_gb300 as wo

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wo.load_library()
    w = WORKLOADS["moe"]
    c = inputs.make_moe_case()
    dt = torch.bfloat16

    def up16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt)

    A = up16(c.A)
    logits = torch.from_numpy(c.logits).to(dev)
    fc1 = wo.pack_experts(torch.from_numpy(c.fc1).to(dev), c.E, 2 * c.I, c.H, 8)
    fc2 = wo.pack_experts(torch.from_numpy(c.fc2).to(dev), c.E, c.H, c.I, 8)
    s1, s2 = up16(c.fc1_scales), up16(c.fc2_scales)
    out = torch.empty((c.T, c.H), dtype=dt, device=dev)
    need = wo.wo_moe_workspace_size(c.T, c.H, c.I, c.E, c.topk)
    workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call(Ain=None):
        wo.wo_moe_ffn(A if Ain is None else Ain, logits, fc1, s1, fc2, s2, out, c.T, c.H, c.I,
                      c.E, c.topk, 0, inputs.BF16, workspace, need, stream)

    with torch.cuda.stream(stream):
        call()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
    torch.cuda.synchronize()
    bytes_per_step = c.weight_bytes
    launches_per_step = 4  # routing, fc1, fc2, combine
    sampler = ClockSampler(local)
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(args.steps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop()
    total_ms = max_over_ranks(ws, start.elapsed_time(end))
    secs = total_ms / 1e3
    value = bytes_per_step * args.steps * ws / secs / 1e9

    # end to end: every step copies its activations and gating logits in from
    # pinned host memory and its output out, on two copy streams with two
    # buffer sets (overlapping the neighbouring steps' kernels, as a serving
    # loop would); events order every buffer's reuse
    hA = torch.empty(A.shape, dtype=dt, pin_memory=True)
    hA.copy_(A.cpu())
    hL = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True)
    hL.copy_(logits.cpu())
    hO = [torch.empty(out.shape, dtype=dt, pin_memory=True) for _ in range(2)]
    dA = [torch.empty_like(A) for _ in range(2)]
    dL = [torch.empty_like(logits) for _ in range(2)]
    dO = [torch.empty_like(out) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_k = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]
    e2e_steps = max(1, min(args.steps, 30))

    def e2e_step(i):
        b = i % 2
        if used[b]:
            s_in.wait_event(ev_k[b])
            stream.wait_event(ev_out[b])
        used[b] = True
        with torch.cuda.stream(s_in):
            dA[b].copy_(hA, non_blocking=True)
            dL[b].copy_(hL, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        with torch.cuda.stream(stream):
            wo.moe_ffn(dA[b], dL[b], fc1, s1, fc2, s2, c.H, c.I, c.E, c.topk, out=dO[b],
                       workspace=workspace, stream=stream)
            ev_k[b].record(stream)
        s_out.wait_event(ev_k[b])
        with torch.cuda.stream(s_out):
            hO[b].copy_(dO[b], non_blocking=True)
            ev_out[b].record(s_out)
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(ws, time.perf_counter() - t0)
    if rank != 0:
        return 0
    hbm_gbs, _, peak_src = measured_peaks()
    achieved = bytes_per_step / (total_ms / args.steps / 1e3) / 1e9
    try:
        sh = kernel_source_hash(["wo_moe.cu", "wo_gemm_tc.cu", "wo_common.cuh", "wo_sm100.cuh"])
    except OSError:
        sh = None
    tr = traffic_from_profile("moe_ffn", sh, "moe") if sh else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w["desc"], "weight_bytes_per_step": bytes_per_step,
                   "l2": f"inputs larger than L2: {bytes_per_step / 1e6:.0f} MB of expert "
                         "weights per step",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "peak_source": f"hbm_gbs ({peak_src})",
                     "traffic": tr["dram_bytes_per_launch"] if tr else None,
                     "kernel": "wo_moe_ffn (routing + fc1 + fc2 + combine, timed together)",
                     "algorithmic_bytes_per_launch": bytes_per_step},
        "e2e": {"value": bytes_per_step * e2e_steps * ws / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": hA.numel() * 2 + hL.numel() * 4,
                "d2h_bytes_per_step": hO[0].numel() * 2,
                "copies": "every step: pinned H2D of its activations and logits, D2H of its "
                          "output, on two copy streams with two buffer sets (overlapping the "
                          "neighbouring steps' kernels)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if ws == 1 and not args.no_cpu_baseline:
        import oracle
        tokens = np.arange(8)
        t0 = time.perf_counter()
        oracle.moe_ffn(c.A, c.act_dtype, c.logits, c.fc1, c.fc1_scales, c.fc2, c.fc2_scales,
                       c.T, c.H, c.I, c.E, c.topk, tokens=tokens)
        dt_s = time.perf_counter() - t0
        ids, _ = oracle.moe_route(c.logits[tokens], c.topk)
        per_expert = c.weight_bytes / c.E
        touched = len(set(ids.reshape(-1).tolist())) * per_expert
        line["cpu_baseline"] = {"value": touched / dt_s / 1e9, "unit": "GB/s",
                                "cores": os.cpu_count() or 1, "kind": "oracle",
                                "sample": f"the first 8 tokens ({touched / 1e6:.0f} MB of the "
                                          f"experts they route to), {dt_s:.2f} s wall"}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------- sub-records of the default run --

L2_BYTES = 129e6
HBM_TARGET, TENSOR_TARGET = 0.70, 0.60  # fractions of the measured peaks

# the decode shapes of 64 MB and more (A16W8 37888x3584 and 3584x18944 at
# m in {1, 4, 16}; the W4A16 131072x2048 lm_head at m = 1): (config, case)
STEADY_DECODE = [(2, 2), (2, 3), (2, 6), (2, 7), (2, 10), (2, 11), (4, 3)]


def upload_case(c, dev):
    import torch

    import weight_only_quantized_fpa_gb300 as wo
    dt = torch.float16 if c.act_dtype == inputs.F16 else torch.bfloat16

    def up16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt)
    B = wo.pack(torch.from_numpy(c.B).to(dev), c.n, c.k, c.bits)
    return dict(c=c, A=up16(c.A), B=B, s=up16(c.scales),
                z=None if c.zeros is None else up16(c.zeros),
                b=None if c.bias is None else up16(c.bias),
                C=torch.empty((c.m, c.n), dtype=dt, device=dev))


def steady_state_case(c, dev, reps=8, repeats=5):
    """One case replayed back to back in one CUDA graph over R copies of its
    weights (R * weight bytes >= 2.5x the L2, so every launch reads its
    weights from HBM): median of `repeats` timed replays of reps * R
    launches.  Returns microseconds per call."""
    import torch

    import weight_only_quantized_fpa_gb300 as wo
    d = upload_case(c, dev)
    R = int(min(64, max(2, np.ceil(2.5 * L2_BYTES / c.weight_bytes))))
    Bs = [d["B"]] + [d["B"].clone() for _ in range(R - 1)]
    Ss = [d["s"]] + [d["s"].clone() for _ in range(R - 1)]
    Zs = [d["z"]] * R if d["z"] is None else [d["z"]] + [d["z"].clone() for _ in range(R - 1)]
    need = wo.wo_workspace_size(c.m, c.n, c.k, c.group_size, c.bits)
    wsb = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call(i):
        wo.wo_gemm(d["A"], Bs[i], Ss[i], Zs[i], d["b"], d["C"], c.m, c.n, c.k, c.group_size,
                   c.bits, c.act_dtype, wsb, wsb.numel(), stream)
    with torch.cuda.stream(stream):
        for i in range(R):
            call(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                for i in range(R):
                    call(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        for _ in range(repeats):
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / (reps * R))
    del g, Bs, Ss, Zs, d
    torch.cuda.empty_cache()
    return statistics.median(times), R


def steady_state_records(dev, specs, hbm_gbs, bf16_tf):
    out = []
    for cfg, i in specs:
        c = inputs.workload_case(cfg, i)
        us, R = steady_state_case(c, dev)
        rec = {"m": c.m, "n": c.n, "k": c.k, "bits": c.bits, "us": us, "weight_copies": R}
        if c.m <= 16:
            gbs = c.weight_bytes / (us / 1e6) / 1e9
            rec.update(gbs=gbs, frac=gbs / hbm_gbs, target=HBM_TARGET,
                       met=gbs / hbm_gbs >= HBM_TARGET)
        else:
            tf = case_flops(c) / (us / 1e6) / 1e12
            rec.update(tflops=tf, frac=tf / bf16_tf,
                       target=TENSOR_TARGET if c.m >= 1024 else None,
                       met=(tf / bf16_tf >= TENSOR_TARGET) if c.m >= 1024 else None)
        out.append(rec)
    return out


def large_m_record(dev, steps, warmup, hbm_gbs, bf16_tf, peak_src):
    """The A16W8 large-m workload (every case once per step, back to back in
    one CUDA graph, CUDA events on the launching stream): TFLOP/s over the
    step and its fraction of the measured dense bf16 peak; per case the
    steady-state TFLOP/s."""
    import torch

    import weight_only_quantized_fpa_gb300 as wo
    cases = workload_cases("w8_large")
    dcs = [upload_case(c, dev) for c in cases]
    need = max(wo.wo_workspace_size(c.m, c.n, c.k, c.group_size, c.bits) for c in cases)
    wsb = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for d in dcs:
            c = d["c"]
            wo.wo_gemm(d["A"], d["B"], d["s"], d["z"], d["b"], d["C"], c.m, c.n, c.k,
                       c.group_size, c.bits, c.act_dtype, wsb, wsb.numel(), stream)
    with torch.cuda.stream(stream):
        step()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flops = sum(case_flops(c) for c in cases)
    tf = flops / (ms / 1e3) / 1e12
    del g, dcs
    torch.cuda.empty_cache()
    try:
        sh = kernel_source_hash(["wo_gemm_tc.cu", "wo_common.cuh", "wo_sm100.cuh"])
    except OSError:
        sh = None
    tr = traffic_from_profile("gemm_tc_kernel", sh, "w8_large") if sh else None
    per_case = steady_state_records(dev, [(3, i) for i in range(len(cases))], hbm_gbs, bf16_tf)
    return {
        "workload": WORKLOADS["w8_large"]["desc"], "unit": "TFLOP/s", "value": tf,
        "ms_per_step": ms, "steps": steps, "warmup": warmup,
        "flops_per_step": flops,
        "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16_tf, "unit": "TFLOP/s",
                     "frac": tf / bf16_tf, "peak_source": f"bf16_tflops burst ({peak_src})",
                     "traffic": tr["dram_bytes_per_launch"] if tr else None,
                     "kernel": "gemm_tc_kernel",
                     "algorithmic_flops_per_launch": flops / len(cases),
                     "timing": f"{len(cases)} GEMM calls per step back to back in one CUDA "
                               "graph; achieved = 2*m*n*k summed over the cases / step time"},
        "target": TENSOR_TARGET,
        "cases_note": "steady state: each case replayed back to back over rotating copies of "
                      "its weights; target applies at m >= 1024",
        "cases": per_case,
    }


def run_ours(args, ws, rank, local):
    import torch

    import weight_only_quantized_fpa_gb300 as wo

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wo.load_library()
    w = WORKLOADS[args.workload]
    cases = workload_cases(args.workload)

    def dt_of(c):
        return torch.float16 if c.act_dtype == inputs.F16 else torch.bfloat16

    def up16(a, c):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt_of(c))

    dev_cases = []
    max_ws = 0
    for c in cases:
        Brm = torch.from_numpy(c.B).to(dev)
        perm = None
        if c.g_idx is not None:  # act-order: codes packed in group-sorted channel order
            perm = wo.act_order_perm(c.g_idx, c.k, c.group_size).to(dev)
            Bp = wo.pack_act_order(Brm, perm, c.n, c.k, c.bits)
            need = wo.wo_act_order_workspace_size(c.m, c.n, c.k, c.group_size, c.bits)
        else:
            Bp = wo.pack(Brm, c.n, c.k, c.bits)
            need = wo.wo_workspace_size(c.m, c.n, c.k, c.group_size, c.bits)
        del Brm
        d = dict(c=c, A=up16(c.A, c), B=Bp, s=up16(c.scales, c), perm=perm,
                 z=None if c.zeros is None else up16(c.zeros, c),
                 b=None if c.bias is None else up16(c.bias, c),
                 C=torch.empty((c.m, c.n), dtype=dt_of(c), device=dev))
        max_ws = max(max_ws, need)
        dev_cases.append(d)
    workspace = torch.zeros(max(max_ws, 256), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel()
    stream = torch.cuda.Stream(device=dev)

    def call(d, A=None, C=None):
        c = d["c"]
        if d["perm"] is not None:
            wo.wo_gemm_act_order(d["A"] if A is None else A, d["B"], d["perm"], d["s"], d["z"],
                                 d["b"], d["C"] if C is None else C, c.m, c.n, c.k,
                                 c.group_size, c.bits, c.act_dtype, workspace, ws_bytes, stream)
            return
        wo.wo_gemm(d["A"] if A is None else A, d["B"], d["s"], d["z"], d["b"],
                   d["C"] if C is None else C, c.m, c.n, c.k, c.group_size, c.bits,
                   c.act_dtype, workspace, ws_bytes, stream)

    # one CUDA graph per step (every case, one kernel each, back to back) for
    # the timed region, and one per case for the per-case breakdown
    graphs = []
    with torch.cuda.stream(stream):
        for d in dev_cases:
            call(d)
        stream.synchronize()
        step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(step_graph, stream=stream):
            for d in dev_cases:
                call(d)
        for d in dev_cases:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(d)
            graphs.append(g)
    torch.cuda.synchronize()

    launches_per_step = sum(case_launches(c) for c in cases)
    bytes_per_step = sum(c.weight_bytes for c in cases)
    flops_per_step = sum(case_flops(c) for c in cases)
    ncase = len(cases)

    sampler = ClockSampler(local)
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step_graph.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(args.steps):
            step_graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop()
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(ws, total_ms)
    secs = total_ms / 1e3

    # per-case breakdown (outside the timed region): each case replayed on its
    # own between the others, so its weights are not in L2; includes the
    # launch gap of a lone graph
    nrep = max(1, min(args.steps, 20))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(ncase + 1)] for _ in range(nrep)]
    with torch.cuda.stream(stream):
        for r in range(nrep):
            for i, g in enumerate(graphs):
                ev[r][i].record(stream)
                g.replay()
            ev[r][ncase].record(stream)
    torch.cuda.synchronize()
    per_case_ms = [statistics.fmean(ev[r][i].elapsed_time(ev[r][i + 1]) for r in range(nrep))
                   for i in range(ncase)]

    if w["unit"] == "GB/s":
        value = bytes_per_step * args.steps * ws / secs / 1e9
    else:
        value = flops_per_step * args.steps * ws / secs / 1e12

    # ---- end to end through the public API with host buffers ----
    # every step: one pinned host -> device copy of all the cases' activations,
    # one wo.gemm per case, one device -> host copy of all the outputs.  As in
    # a serving loop the copies run on their own streams with two buffer sets:
    # step i's input copy overlaps step i - 1's kernels and step i's output
    # copy step i + 1's kernels; events order every buffer's reuse.
    a_sizes = [d["A"].numel() for d in dev_cases]
    c_sizes = [d["C"].numel() for d in dev_cases]
    a_dt, c_dt = dev_cases[0]["A"].dtype, dev_cases[0]["C"].dtype
    host_A = torch.empty(sum(a_sizes), dtype=a_dt, pin_memory=True)
    host_C = [torch.empty(sum(c_sizes), dtype=c_dt, pin_memory=True) for _ in range(2)]
    dev_A = [torch.empty(sum(a_sizes), dtype=a_dt, device=dev) for _ in range(2)]
    dev_C = [torch.empty(sum(c_sizes), dtype=c_dt, device=dev) for _ in range(2)]
    a_views, c_views = [[], []], [[], []]
    off_a = off_c = 0
    for d, na, nc in zip(dev_cases, a_sizes, c_sizes):
        host_A[off_a:off_a + na].copy_(d["A"].reshape(-1).cpu())
        for b in range(2):
            a_views[b].append(dev_A[b][off_a:off_a + na].view(d["A"].shape))
            c_views[b].append(dev_C[b][off_c:off_c + nc].view(d["C"].shape))
        off_a += na
        off_c += nc
    h2d = host_A.numel() * host_A.element_size()
    d2h = host_C[0].numel() * host_C[0].element_size()
    e2e_steps = max(1, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]   # set b's input copy done
    ev_k = [torch.cuda.Event() for _ in range(2)]    # set b's kernels done
    ev_out = [torch.cuda.Event() for _ in range(2)]  # set b's output copy done
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        if used[b]:
            s_in.wait_event(ev_k[b])      # the kernels two steps back read dev_A[b]
            stream.wait_event(ev_out[b])  # and their outputs left dev_C[b]
        used[b] = True
        with torch.cuda.stream(s_in):
            dev_A[b].copy_(host_A, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        with torch.cuda.stream(stream):
            for d, Av, Cv in zip(dev_cases, a_views[b], c_views[b]):
                c = d["c"]
                if d["perm"] is not None:
                    wo.gemm_act_order(Av, d["B"], d["perm"], d["s"], c.n, c.k, c.bits,
                                      c.group_size, zeros=d["z"], bias=d["b"], out=Cv,
                                      workspace=workspace, stream=stream)
                    continue
                wo.gemm(Av, d["B"], d["s"], c.n, c.k, c.bits, group_size=c.group_size,
                        zeros=d["z"], bias=d["b"], out=Cv, workspace=workspace,
                        stream=stream)
            ev_k[b].record(stream)
        s_out.wait_event(ev_k[b])
        with torch.cuda.stream(s_out):
            host_C[b].copy_(dev_C[b], non_blocking=True)
            ev_out[b].record(s_out)
    for i in range(min(3, e2e_steps)):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(ws, time.perf_counter() - t0)
    if w["unit"] == "GB/s":
        e2e_val = bytes_per_step * e2e_steps * ws / e2e_s / 1e9
    else:
        e2e_val = flops_per_step * e2e_steps * ws / e2e_s / 1e12

    if rank != 0:
        return 0

    hbm_gbs, bf16_tf, peak_src = measured_peaks()
    # the step graph holds only this library's kernels, the GEMM kernel of
    # each case (plus its prepasses: act-order gather, fp16 copy of bf16 A),
    # back to back: the algorithmic bytes (or flops) over the step time
    kern_ms = total_ms / args.steps
    if w["unit"] == "GB/s":
        achieved = bytes_per_step / (kern_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "peak_source": f"hbm_gbs ({peak_src})"}
    else:
        achieved = flops_per_step / (kern_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16_tf, "unit": "TFLOP/s",
                "frac": achieved / bf16_tf, "peak_source": f"bf16_tflops burst ({peak_src})"}
    kname, src = dominant_kernel(wo, cases, w["unit"] != "GB/s")
    try:
        sh = kernel_source_hash(src)
    except OSError:
        sh = None
    tr = traffic_from_profile(kname, sh, args.workload) if sh else None
    roof["traffic"] = tr["dram_bytes_per_launch"] if tr else None
    if w["unit"] == "GB/s":
        roof["algorithmic_bytes_per_launch"] = bytes_per_step / ncase
    else:
        roof["algorithmic_flops_per_launch"] = flops_per_step / ncase
    roof["kernel"] = kname
    roof["timing"] = (f"{ncase} GEMM calls ({launches_per_step} launches) per step back to "
                      "back in one CUDA graph; achieved = "
                      "algorithmic bytes (or flops) per step / step time")

    line = {
        "metric": METRIC, "value": value, "unit": w["unit"], "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": w["desc"], "cases": ncase,
                   "weight_bytes_per_step": bytes_per_step,
                   "l2": ("inputs larger than L2: every case has its own weights "
                          f"({bytes_per_step / 1e6:.0f} MB per step)") if bytes_per_step > 129e6
                         else (f"working set {bytes_per_step / 1e6:.2f} MB fits in L2 and is not "
                               "flushed: a latency-bound parity case"),
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": roof,
        "cases_note": "per case: replayed alone between the other cases (cold L2), "
                      "launch gap of a lone graph included",
        "cases": [{"m": c.m, "n": c.n, "k": c.k, "us": ms * 1e3,
                   ("gbs" if w["unit"] == "GB/s" else "tflops"):
                       (c.weight_bytes / (ms / 1e3) / 1e9) if w["unit"] == "GB/s"
                       else case_flops(c) / (ms / 1e3) / 1e12}
                  for c, ms in zip(cases, per_case_ms)],
        "e2e": {"value": e2e_val, "unit": w["unit"], "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": "every step: one pinned H2D of its inputs, one D2H of its outputs, on "
                          "two copy streams with two buffer sets (overlapping the neighbouring "
                          "steps' kernels)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if args.workload == "w8_decode" and not args.no_sub_records:
        # the other half of the metric (TFLOP/s at m >= 64) and the per-shape
        # steady state of the >= 64 MB decode shapes, timed after the main
        # region (they do not enter `value`)
        line["large_m"] = large_m_record(dev, max(5, min(args.steps, 20)), max(3, args.warmup),
                                         hbm_gbs, bf16_tf, peak_src)
        line["steady_state"] = {
            "note": "each case replayed back to back in one CUDA graph over rotating copies of "
                    "its weights (>= 2.5x L2), CUDA events on the launching stream; frac of "
                    "the measured HBM copy bandwidth, target 0.70",
            "cases": steady_state_records(dev, STEADY_DECODE, hbm_gbs, bf16_tf)}
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cases, w["unit"])
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.profile_case is not None:
        return run_profile_case(args)
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        rc = run_reference(args, ws, rank)
    elif args.workload == "moe":
        rc = run_moe(args, ws, rank, local)
    elif args.workload == "embed":
        rc = run_embed(args, ws, rank, local)
    else:
        rc = run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
