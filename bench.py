#!/usr/bin/env python3
"""Muon step benchmark on GB300 (one process per GPU; replicas only, no collective).

Default workload: one Qwen3-4B-shaped transformer layer (q 4096x2560, k/v 1024x2560,
o 2560x4096, gate/up 9728x2560, down 2560x9728), gradients bf16 N(0, 1e-3),
momentum and fp32 master weights N(0, 0.02), mu 0.95 Nesterov, lr 0.02, 5 quintic
Newton-Schulz iterations.  A step is one muon_step over the 7 matrices.

Prints ONE JSON line on rank 0.  --impl reference times the fp64 CPU oracle on the
host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon step matrices/s and NS TFLOP/s (% BF16 peak) at Qwen3-4B shapes, 1 GB300"
QWEN3_4B_LAYER = [("q_proj", 4096, 2560), ("k_proj", 1024, 2560), ("v_proj", 1024, 2560),
                  ("o_proj", 2560, 4096), ("gate_proj", 9728, 2560), ("up_proj", 9728, 2560),
                  ("down_proj", 2560, 9728)]
WORKLOAD = ("qwen3-4b-layer: q 4096x2560, k/v 1024x2560, o 2560x4096, gate/up 9728x2560, "
            "down 2560x9728; G bf16 N(0,1e-3), M and W fp32 N(0,0.02); mu 0.95 Nesterov, lr 0.02, "
            "wd 0, 5 NS iterations (3.4445, -4.7750, 2.0315)")
LR, MU, WD, NS_STEPS = 0.02, 0.95, 0.0, 5
NS_COEFFS = (3.4445, -4.7750, 2.0315)
# Newton-Schulz coefficients: "fixed" (the configuration's (a, b, c) every
# iteration) or "minimax" (per-iteration schedule, see --ns-schedule); set by main()
NS_SCHEDULE = {"kind": "fixed", "lower": 1e-3, "safety": 1.05}
# Newton-Schulz method: "standard" (the iteration on X) or "gram" (on X X^T); set by main()
NS_METHOD = "standard"
G_SIGMA, W_SIGMA, M_SIGMA = 1e-3, 0.02, 0.02


def ns_flops(rows, cols, steps=None):
    """(nominal, algorithmic) Newton-Schulz flops of one rows x cols matrix."""
    steps = NS_STEPS if steps is None else steps
    m, n = min(rows, cols), max(rows, cols)
    nominal = steps * (4 * m * m * n + 2 * m ** 3)
    algorithmic = steps * (m * (m + 1) * n + 2 * m ** 3 + 2 * m * m * n)
    return nominal, algorithmic


def ns_executed_flops(rows, cols, steps=None, bm=128, bn=256, bk=64, small=False):
    """Flops the tensor cores execute.  Grouped GEMMs: whole 128x256 tiles touching
    the upper triangle (GRAM, POLY) or covering the output (UPDATE), k rounded up to
    64.  The small-matrix kernel (m <= 128): every product on 128 x 128 tiles, X in
    128-column chunks (Gram K and UPDATE N rounded up to 128)."""
    steps = NS_STEPS if steps is None else steps
    m, n = min(rows, cols), max(rows, cols)
    cd = lambda a, b: -(-a // b)
    if small and NS_METHOD == "gram":
        # Gram and U = R X0 (high and low parts of R) over the chunks; per iteration
        # A A, Q A, Q R and (Q A) Q as three bf16 products each (the last iteration
        # skips Q A and (Q A) Q)
        npad = cd(n, 128) * 128
        sq = 3 * 2 * 128 ** 3
        return 2 * 128 * 128 * npad + 2 * 2 * 128 * 128 * npad + sq * (4 * steps - 2)
    if small:
        npad = cd(n, 128) * 128
        return steps * (2 * 128 * 128 * npad + 2 * 128 ** 3 + 2 * 128 * 128 * npad)
    sym = sum(min(cd(m, bm), (bj * bn + bn - 1) // bm + 1) for bj in range(cd(m, bn)))
    gram = sym * bm * bn * cd(n, bk) * bk * 2
    poly = sym * bm * bn * cd(m, bk) * bk * 2
    upd = cd(m, bm) * cd(n, bn) * bm * bn * cd(m, bk) * bk * 2
    return steps * (gram + poly + upd)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values):
    """Element-wise maximum of per-rank floats over the process group (identity on one
    rank); CUDA tensors under NCCL, CPU tensors under gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(units_per_rank, world, ms):
    """Units of all ranks per second, over the slowest rank's time per step."""
    return units_per_rank * world / (ms / 1000.0)


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# CPU oracle timing (bench's cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(spec, n_sample):
    """Inputs of an evenly spaced sample of the workload's logical matrices, generated on
    the CPU from the same seeded streams the device fill uses (bit-identical values)."""
    import synth
    flat = [(i, j, r, c) for i, (r, c, k) in enumerate(spec["tensors"]) for j in range(k)]
    n = min(n_sample, len(flat))
    picks = [flat[(q * len(flat)) // n] for q in range(n)]
    out = []
    for i, j, r, c in picks:
        start = j * r * c
        W = synth.tensor(synth.SEED, synth.stream_id(i, synth.ROLE_W), 0, (r, c), spec["w_sigma"], spec["w_dtype"],
                         start=start)
        if spec["m_sigma"] > 0:
            M = synth.tensor(synth.SEED, synth.stream_id(i, synth.ROLE_M), 0, (r, c), spec["m_sigma"], synth.F32,
                             start=start)
        else:
            M = np.zeros((r, c), dtype=np.float32)
        G = synth.tensor(synth.SEED, synth.stream_id(i, synth.ROLE_G), 0, (r, c), spec["g_sigma"], spec["g_dtype"],
                         start=start)
        out.append((synth.as_f64(W, spec["w_dtype"]), M, synth.as_f64(G, spec["g_dtype"])))
    return out


def oracle_coeffs():
    """The oracle's coefficients for the configured schedule."""
    import oracle
    if NS_SCHEDULE["kind"] == "minimax":
        return oracle.polar_express_schedule(NS_STEPS, NS_SCHEDULE["lower"], NS_SCHEDULE["safety"])[0]
    return oracle.DEFAULT_COEFFS


def oracle_step(sample):
    import oracle
    co = oracle_coeffs()
    for W, M, G in sample:
        oracle.muon_matrix_step(W, M, G, LR, MU, True, WD, NS_STEPS, co, method=NS_METHOD)


def schedule_config():
    """The --ns-schedule and --ns-method choices as both arms state them in their config."""
    if NS_SCHEDULE["kind"] != "minimax":
        out = {"kind": "fixed", "coeffs": [3.4445, -4.7750, 2.0315]}
    else:
        out = {"kind": "minimax", "lower": NS_SCHEDULE["lower"], "safety": NS_SCHEDULE["safety"]}
    if NS_METHOD != "standard":
        out["method"] = NS_METHOD
    return out


def spec_bytes(spec):
    """Bytes of W, M and G of one step of a workload."""
    import synth
    size = {synth.F32: 4, synth.BF16: 2}
    return sum(k * r * c * (size[spec["w_dtype"]] + 4 + size[spec["g_dtype"]]) for r, c, k in spec["tensors"])


def arm_config(spec, world):
    """The config object of the JSON line, the same for the GPU arm and the reference arm."""
    elems = sum(k * r * c for r, c, k in spec["tensors"])
    return {"workload": spec["desc"], "matrices_per_step": sum(k for _, _, k in spec["tensors"]),
            "elements_per_step": elems, "ns_steps": NS_STEPS, "ns_schedule": schedule_config(),
            "parallelism": f"replicas{world}",
            "l2": f"inputs {spec_bytes(spec) / 1e9:.2f} GB per step vs the 129 MB L2"}


OFFLOAD_DESC = ("36 Qwen3-4B layers (3.63B Muon parameters) with G bf16 and fp32 M in pinned host memory; "
                "128 MiB buckets, three staging slots (upload, compute and writeback of three buckets overlap); "
                "host-blocking step (drained before return)")


def offload_config(world, zero_copy=False):
    return {"workload": OFFLOAD_DESC, "matrices_per_step": 36 * len(QWEN3_4B_LAYER), "ns_steps": NS_STEPS,
            "ns_schedule": schedule_config(), "parallelism": f"replicas{world}",
            "offload_mode": "zero-copy (kernels read and write the pinned host buffers)" if zero_copy
            else "staged (copy engines into device slots)"}


def set_schedule(nsm, plan):
    """Applies --ns-schedule to a plan; returns its description for the JSON line."""
    if NS_SCHEDULE["kind"] != "minimax":
        return {"kind": "fixed", "coeffs": [3.4445, -4.7750, 2.0315]}
    co, err = nsm.muon_polar_express_coefficients(NS_STEPS, NS_SCHEDULE["lower"], NS_SCHEDULE["safety"])
    nsm.muon_set_ns_schedule(plan, co)
    return {"kind": "minimax (per-iteration odd quintic closest to 1 on the singular-value interval)",
            "lower": NS_SCHEDULE["lower"], "safety": NS_SCHEDULE["safety"],
            "coeffs": [[round(v, 6) for v in t] for t in co], "worst_case_error_after_each": err}


# matrices the CPU leg times per workload: the whole layer, or a bounded sample
CPU_SAMPLE = {"layer": 7, "single": 1, "heads": 64, "experts": 16, "offload": 7}


def cpu_baseline_leg(name, min_seconds=10.0):
    spec = workload_spec("layer" if name == "offload" else name)
    sample = oracle_sample(spec, CPU_SAMPLE[name])
    reps, dt = 0, 0.0
    t0 = time.perf_counter()
    while reps == 0 or dt < min_seconds:
        oracle_step(sample)
        reps += 1
        dt = time.perf_counter() - t0
    n = reps * len(sample)
    what = ("the 7 matrices of one Qwen3-4B layer (the offload step has the same matrices)"
            if name in ("layer", "offload") else
            "the workload's one matrix" if len(sample) == 1 else
            f"{len(sample)} evenly spaced matrices of the workload")
    return {"value": n / dt, "unit": "matrices/s", "cores": cores_used(), "kind": "oracle",
            "sample": f"{what}, {reps} pass(es), {dt:.1f} s; numpy fp64 with OpenBLAS threads"}


# seconds of oracle work the reference arm's timed steps may take in total
REF_TIMED_BUDGET_S = 120.0


def run_reference(args):
    """The oracle, as it stands, on the host cores: the reference arm of this bench.

    Each timed step runs the oracle on a sample of the workload's matrices, the
    cheapest first, as many as fit in REF_TIMED_BUDGET_S / steps at the rate the
    warm-up measured (at least one), so the run ends in a few minutes for any
    --steps.  The fp64 flop rate of those steps, divided into the workload's
    Newton-Schulz flops, gives the workload's matrices/s.
    """
    rank, world, _ = dist_env()
    if rank != 0:
        return
    name = args.workload
    spec = workload_spec("layer" if name == "offload" else name)
    sample = oracle_sample(spec, CPU_SAMPLE[name])
    flops = [ns_flops(*W.shape)[1] for (W, _, _) in sample]
    order = sorted(range(len(sample)), key=lambda i: flops[i])
    t0 = time.perf_counter()
    for _ in range(args.warmup):            # warm-up on the cheapest sampled matrix
        oracle_step([sample[order[0]]])
    rate = max(args.warmup, 1) * flops[order[0]] / max(time.perf_counter() - t0, 1e-9)
    per_step = max(0.5, REF_TIMED_BUDGET_S / max(args.steps, 1))
    picked, est = [], 0.0
    for i in order:
        if picked and est + flops[i] / rate > per_step:
            break
        picked.append(i)
        est += flops[i] / rate
    timed = [sample[i] for i in picked]
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(timed)
    dt = time.perf_counter() - t0
    measured = args.steps * sum(flops[i] for i in picked) / dt          # fp64 flop/s of the oracle
    if name == "offload":
        work = [(r, c) for _ in range(36) for (_, r, c) in QWEN3_4B_LAYER]
    else:
        work = [(r, c) for (r, c, k) in spec["tensors"] for _ in range(k)]
    step_s = sum(ns_flops(r, c)[1] for r, c in work) / measured          # one whole workload step
    value = len(work) / step_s
    sample_ms = 1000 * dt / args.steps
    sample_desc = (f"each timed step runs the oracle on {len(timed)} of the workload's matrices "
                   f"(the cheapest of an evenly spaced sample of {len(sample)}, {per_step:.1f} s per step at "
                   f"most); matrices/s of the whole workload from the measured fp64 flop rate "
                   f"({measured / 1e9:.2f} GFLOP/s of Newton-Schulz work), extrapolated by flop ratio")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "matrices/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sample_ms,
        "ms_per_step_note": ("wall time of one timed step, i.e. of the oracle on the timed sample; the "
                             "whole workload's step, extrapolated by flop ratio, is "
                             "ms_per_step_whole_workload_extrapolated"),
        "ms_per_step_whole_workload_extrapolated": 1000 * step_s,
        "matrices_per_timed_step": len(timed),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": offload_config(world) if name == "offload" else arm_config(spec, world),
        "cpu_baseline": {"value": value, "unit": "matrices/s", "cores": cores_used(), "kind": "oracle",
                         "sample": sample_desc},
        "e2e": {"value": value, "unit": "matrices/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def mhz(s):
            try:
                return float(s.split()[0])
            except Exception:
                return float("nan")
        sm = [mhz(r[1]) for r in rows]
        mx = [mhz(r[2]) for r in rows]
        power = [mhz(r[3]) for r in rows]
        loaded = [r for r, p in zip(rows, power) if p == p and p > 300.0] or rows
        sm_loaded = [mhz(r[1]) for r in loaded]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in loaded:
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm_loaded)), "sm_max_mhz": float(np.nanmax(mx)),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": float(np.nanmax(power))}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
# DRAM bytes (read + write) per launch from one ncu capture each, valid only for the
# kernel sources they were taken on (the bench reports null once their digest
# moves).  The commands and per-launch tables are in profiles/.
#  - ns_gemm on the default workload: the mean over the 15 launches of one step
#    (profiles/ns_gemm_qwen3_4b_layer.md).
#  - the small-matrix kernels on 128 x 2560 heads (momentum kernel first): one
#    launch over 7 layers (336 matrices), per matrix; a full launch scales by the
#    matrices it holds (profiles/ns_gram_per_head_qkv.md, ns_small_per_head_qkv.md).
GEMM_SOURCES = ['newton_schulz_muon_gb300/csrc/ns_gemm.cu', 'newton_schulz_muon_gb300/csrc/device.cuh', 'newton_schulz_muon_gb300/csrc/kernels.h', 'newton_schulz_muon_gb300/csrc/epilogue.cuh']
GRAM_SOURCES = ['newton_schulz_muon_gb300/csrc/ns_gram.cu', 'newton_schulz_muon_gb300/csrc/small_common.cuh', 'newton_schulz_muon_gb300/csrc/device.cuh', 'newton_schulz_muon_gb300/csrc/kernels.h', 'newton_schulz_muon_gb300/csrc/epilogue.cuh', 'newton_schulz_muon_gb300/csrc/momentum.cuh']
SMALL_SOURCES = ['newton_schulz_muon_gb300/csrc/ns_small.cu', 'newton_schulz_muon_gb300/csrc/small_common.cuh', 'newton_schulz_muon_gb300/csrc/device.cuh', 'newton_schulz_muon_gb300/csrc/kernels.h', 'newton_schulz_muon_gb300/csrc/epilogue.cuh', 'newton_schulz_muon_gb300/csrc/momentum.cuh']
NS_GEMM_TRAFFIC = {"bytes_per_launch": 349.8e6, "sources_sha256_16": "fedaaee9110f4a6f"}
HEAD_TRAFFIC = {
    "gram": {"bytes_per_matrix": (868.6e6 + 385.4e6) / 336, "sources_sha256_16": "0f481e2ae9140ef6"},
    "standard": {"bytes_per_matrix": (993.6e6 + 846.1e6) / 336, "sources_sha256_16": "1a27241ab7278f8c"},
}


def sources_digest(files):
    import hashlib
    h = hashlib.sha256()
    root = os.path.dirname(os.path.abspath(__file__))
    for f in files:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ns_gemm_traffic():
    if sources_digest(GEMM_SOURCES) != NS_GEMM_TRAFFIC["sources_sha256_16"]:
        return None
    return NS_GEMM_TRAFFIC["bytes_per_launch"]


def head_traffic(method, n_matrices):
    """DRAM bytes of one small-matrix launch over n 128 x 2560 heads (momentum kernel
    first), scaled from the 7-layer capture; None once the kernel's sources moved."""
    t = HEAD_TRAFFIC[method]
    if sources_digest(GRAM_SOURCES if method == "gram" else SMALL_SOURCES) != t["sources_sha256_16"]:
        return None
    return t["bytes_per_matrix"] * n_matrices


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def launches_per_step(nsm, plan, info, ns_only=False):
    """Kernels one step launches: momentum and norm per bucket (unless the
    small-matrix kernel computes the momentum), then one small-matrix
    Newton-Schulz kernel or three GEMMs per iteration.  ns_only: the
    Newton-Schulz launches alone."""
    n = 0
    for b in range(info.n_buckets):
        bi = nsm.muon_get_bucket_info(plan, b)
        ns = 1 if bi.ns_single_kernel else 3 * NS_STEPS
        momentum = 0 if (bi.momentum_in_ns_kernel and NS_STEPS > 0) else 2
        n += ns + (0 if ns_only else momentum)
    return n


def ns_kernel_name(nsm, plan, info):
    single = [nsm.muon_get_bucket_info(plan, b).ns_single_kernel for b in range(info.n_buckets)]
    if all(single) and NS_METHOD == "gram":
        return ("ns_gram_kernel (bf16 X, the iteration on X X^T with split-bf16 128x128 products, "
                "X read twice, with the fused weight update)")
    if all(single):
        return "ns_small_kernel (bf16, every iteration in one launch, with the fused weight update)"
    if not any(single):
        return "ns_gemm_kernel (bf16, with the fused weight update)"
    return "ns_gemm_kernel and ns_small_kernel (bf16, with the fused weight update)"


def choose_bf16_peak(peaks, peak_kind, clocks, timed_s):
    """The bf16 denominator: the burst figure for a kernel that ran at full clock in
    a short timed region, the sustained one where the power cap held the clock down
    or the timed region lasted seconds (the sustained figure was taken over a 4 s
    loop).  Returns (TFLOP/s, description)."""
    sustained = "sw_power_cap" in clocks.get("reasons", []) or timed_s >= 2.0
    if sustained:
        return (peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
                f"{peak_kind} bf16 sustained (power cap active or a timed region of seconds: {timed_s:.2f} s)")
    return peaks["bf16_tflops"], f"{peak_kind} bf16 burst (no power cap seen, timed region {timed_s:.2f} s)"


def ns_compulsory_bytes(tensors, w_sizes, g_sizes, momentum_fused, method="standard"):
    """Bytes the single-launch small-matrix kernel must move through HBM: the
    weights read and written once, plus X0 read once (bf16) or, when the kernel
    computes the momentum itself, G read once and M read and written once.  The
    gram method reads X0 a second time for U = R X0 (and, computing the momentum
    itself, writes X0 once for that)."""
    total = 0
    for (r, c, k), ws, gs in zip(tensors, w_sizes, g_sizes):
        e = k * r * c
        total += 2 * e * ws + (e * (gs + 8) if momentum_fused else e * 2)
        if method == "gram":
            total += e * (4 if momentum_fused else 2)
    return total


def hbm_binds(nbytes, flops, hbm_gbs, tensor_tflops):
    """True when moving `nbytes` at the HBM peak takes longer than `flops` at the
    tensor peak: the roofline of that kernel is HBM."""
    return nbytes / (hbm_gbs * 1e9) > flops / (tensor_tflops * 1e12)


def tf32_peak(bf16_peak):
    """The 3xTF32 mode's fallback denominator: kind::tf32 products run at half the
    kind::f16 rate per SM on this part (a probe measured 4096 flop/clk/SM against
    8192), so the measured bf16 figure times 0.5."""
    return 0.5 * bf16_peak


def measure_tf32_gemm_tflops(n=8192, iters=20):
    """cuBLAS's tf32 GEMM rate on this GPU, timed in this run: torch.matmul of two
    n x n fp32 matrices with TF32 tensor cores allowed, CUDA events around `iters`
    products after three warm-up ones.  It is measured like the bf16 figure of the
    peaks file (a library GEMM, burst), for a dtype that file does not cover."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        g = torch.Generator(device="cuda").manual_seed(0)
        a = torch.randn(n, n, device="cuda", generator=g)
        b = torch.randn(n, n, device="cuda", generator=g)
        c = torch.empty(n, n, device="cuda")
        for _ in range(3):
            torch.matmul(a, b, out=c)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(iters):
            torch.matmul(a, b, out=c)
        e1.record()
        torch.cuda.synchronize()
        sec = e0.elapsed_time(e1) * 1e-3 / iters
        del a, b, c
        return 2.0 * n ** 3 / sec / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def roofline_entry(nsm, plan, info, tf32, hbm_bound, ns_ms, ns_launches, algorithmic, executed, ns_bytes,
                   peak_tf, peak_name, peaks, bf16_sustained, traffic,
                   bytes_counted="compulsory bytes: inputs read once, weights read and written once"):
    """The roofline object of the Newton-Schulz phase's dominant kernel, per launch.

    A tensor-bound kernel is measured on the flops its tensor cores execute (whole
    tiles, the symmetric products' upper tiles only), so ``frac`` cannot pass 1 on
    work the kernel skips; the algorithmic count (upper-triangle Gram, full A A and
    B X) is reported beside it.  3xTF32 executes three tf32 products per product."""
    mult = 3 if tf32 else 1
    sec = ns_ms * 1e-3
    exe_tf = executed * mult / sec / 1e12
    alg_tf = algorithmic * mult / sec / 1e12
    out = {"kernel": ns_kernel_name(nsm, plan, info) + (", 3xTF32" if tf32 else ""),
           "per_launch_ms": ns_ms / ns_launches}
    if hbm_bound:
        gbs = ns_bytes / sec / 1e9
        out.update({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"], "traffic": traffic,
                    "peak_kind": "measured HBM copy bandwidth",
                    "algorithmic_bytes_per_launch": ns_bytes / ns_launches,
                    "bytes_counted": bytes_counted,
                    "tensor_frac": exe_tf / peak_tf, "tensor_frac_algorithmic": alg_tf / peak_tf,
                    "tensor_peak_kind": peak_name})
    else:
        out.update({"bound": "tensor", "achieved": exe_tf, "peak": peak_tf, "unit": "TFLOP/s",
                    "frac": exe_tf / peak_tf, "traffic": traffic, "peak_kind": peak_name,
                    "flops_counted": "executed (whole tiles; upper tiles of X X^T and A A)",
                    "executed_flops_per_launch": executed * mult / ns_launches,
                    "achieved_algorithmic": alg_tf, "frac_algorithmic": alg_tf / peak_tf,
                    "algorithmic_flops_per_launch": algorithmic * mult / ns_launches})
        if not tf32:
            out["frac_of_burst"] = exe_tf / peaks["bf16_tflops"]
            out["frac_of_sustained"] = exe_tf / bf16_sustained
            out["frac_algorithmic_of_burst"] = alg_tf / peaks["bf16_tflops"]
    out["traffic_unit"] = "bytes per launch (dram read + write, one ncu capture)"
    return out


def workload_spec(name, layers=None):
    """Tensors (rows, cols, count), dtypes, distributions and bucket cap of a workload.
    `layers` shortens the per-head and expert workloads (for profiling captures)."""
    import synth
    if name == "layer":
        return dict(desc=WORKLOAD, tensors=[(r, c, 1) for _, r, c in QWEN3_4B_LAYER], g_dtype=synth.BF16,
                    g_sigma=G_SIGMA, w_dtype=synth.F32, w_sigma=W_SIGMA, m_sigma=M_SIGMA, cap=512 << 20)
    if name == "single":
        return dict(desc="single 256x512 matrix: W fp32 N(0,0.02), G fp32 N(0,1), M zero; mu 0.95 Nesterov, "
                         "lr 0.02, wd 0, 5 NS iterations", tensors=[(256, 512, 1)], g_dtype=synth.F32,
                    g_sigma=1.0, w_dtype=synth.F32, w_sigma=W_SIGMA, m_sigma=0.0, cap=512 << 20)
    if name == "heads":
        nl = layers or 36
        return dict(desc=f"per-head Muon on fused interleaved QKV [6144, 2560] x {nl} layers: {48 * nl} logical "
                         "128x2560 matrices in one batch; G bf16 N(0,1e-3), M and W fp32 N(0,0.02)",
                    tensors=[(128, 2560, 48)] * nl, g_dtype=synth.BF16, g_sigma=G_SIGMA, w_dtype=synth.F32,
                    w_sigma=W_SIGMA, m_sigma=M_SIGMA, cap=0)
    if name == "experts":
        nl = layers or 48
        t = []
        for _ in range(nl):
            t += [(768, 2048, 128), (768, 2048, 128), (2048, 768, 128)]
        return dict(desc=f"MoE experts of a 30B-A3B shape: gate/up [128,768,2048], down [128,2048,768] x {nl} "
                         f"layers ({384 * nl} matrices); G bf16 N(0,1e-3), M zero, W bf16 N(0,0.02); 512 MiB buckets",
                    tensors=t, g_dtype=synth.BF16, g_sigma=G_SIGMA, w_dtype=synth.BF16, w_sigma=W_SIGMA,
                    m_sigma=0.0, cap=512 << 20)
    raise ValueError(name)


def library_step(torch, W, M, G, coeffs, lr=LR, mu=MU, wd=WD, eps=1e-7):
    """The same Muon step written the way the pages run it, with library kernels: a
    Python loop over the workload's tensors, each a batch of same-shape logical
    matrices, doing fp32 EMA momentum with Nesterov look-ahead, the Frobenius norm, the
    bf16 cast and the quintic iterations as batched bf16 GEMMs (cuBLAS on the GPU, fp32
    accumulation; b A + c A A and a X + B X through the GEMMs' beta), then the scaled
    weight update.  A timing reference for the hand-written kernels, not a product
    path."""
    for w, m, g in zip(W, M, G):
        m.mul_(mu).add_(g, alpha=1.0 - mu)
        v = m * mu
        v.add_(g, alpha=1.0 - mu)
        tall = v.shape[-2] > v.shape[-1]
        x = v.mT if tall else v
        nrm = torch.linalg.vector_norm(x, dim=(-2, -1), keepdim=True).add_(eps)
        x = (x / nrm).to(torch.bfloat16)
        for a, b, c in coeffs:
            A = torch.bmm(x, x.mT)
            B = torch.baddbmm(A, A, A, beta=b, alpha=c)
            x = torch.baddbmm(x, B, x, beta=a)
        u = x.mT if tall else x
        scale = math.sqrt(max(1.0, w.shape[-2] / w.shape[-1]))
        if wd:
            w.mul_(1.0 - lr * wd)
        w.add_(u.to(w.dtype), alpha=-lr * scale)


def library_step_ms(torch, W, M, G, steps, coeffs):
    """CUDA-event time of library_step (one untimed step first); W and M are left changed."""
    library_step(torch, W, M, G, coeffs)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        library_step(torch, W, M, G, coeffs)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_gpu(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from newton_schulz_muon_gb300.build import build
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
    import newton_schulz_muon_gb300 as nsm
    import synth

    spec = workload_spec(args.workload, args.layers)
    tensors = spec["tensors"]
    shapes = [(r, c, k, 0) for (r, c, k) in tensors]
    tf32 = args.ns_precision == "tf32x3"
    cfg = nsm.muon_config_default(timing=1, grad_dtype=spec["g_dtype"], param_dtype=spec["w_dtype"],
                                  ns_precision=nsm.MUON_NS_TF32X3 if tf32 else nsm.MUON_NS_BF16,
                                  ns_momentum_fused=1 if args.momentum == "fused" else 0,
                                  ns_method=nsm.MUON_NS_METHOD_GRAM if NS_METHOD == "gram"
                                  else nsm.MUON_NS_METHOD_STANDARD)
    cap = spec["cap"] if args.bucket_cap_mib is None else int(args.bucket_cap_mib) << 20
    plan = nsm.muon_plan(shapes, bucket_cap_bytes=cap, config=cfg)
    info = nsm.muon_get_plan_info(plan)
    momentum_fused = all(nsm.muon_get_bucket_info(plan, b).momentum_in_ns_kernel for b in range(info.n_buckets))
    ws = nsm.allocate_workspace(plan)
    schedule = set_schedule(nsm, plan)
    tdt = {synth.F32: torch.float32, synth.BF16: torch.bfloat16}
    W, M, G = [], [], []
    for i, (r, c, k) in enumerate(tensors):
        w = torch.empty((k, r, c), dtype=tdt[spec["w_dtype"]], device="cuda")
        mm = torch.zeros((k, r, c), dtype=torch.float32, device="cuda")
        g = torch.empty((k, r, c), dtype=tdt[spec["g_dtype"]], device="cuda")
        synth.fill_normal_cuda(w, synth.SEED, synth.stream_id(i, synth.ROLE_W), 0, spec["w_sigma"])
        if spec["m_sigma"] > 0:
            synth.fill_normal_cuda(mm, synth.SEED, synth.stream_id(i, synth.ROLE_M), 0, spec["m_sigma"])
        synth.fill_normal_cuda(g, synth.SEED, synth.stream_id(i, synth.ROLE_G), 0, spec["g_sigma"])
        W.append(w); M.append(mm); G.append(g)
    stream = torch.cuda.current_stream()
    n_mats = int(info.n_matrices)

    def step(grads=None):
        nsm.muon_step(plan, W, grads if grads is not None else G, M, LR, MU, True, WD, NS_STEPS, stream)

    for _ in range(args.warmup):
        step()
    st, nf = nsm.muon_sync(plan, stream)
    if st != nsm.MUON_OK:
        raise RuntimeError(f"device status {st} after warm-up")

    # ---- timed region: K steps, inputs larger than L2 ----
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks([ms])[0]
    st, nf = nsm.muon_sync(plan, stream)
    if st != nsm.MUON_OK:
        raise RuntimeError(f"device status {st} after the timed region")
    value = whole_job_rate(n_mats, world, ms)

    # ---- per-phase times (CUDA events inside the library, one step at a time) ----
    prep, nsms = [], []
    for _ in range(5):
        step()
        s = nsm.muon_get_stats(plan)
        prep.append(s.prep_ms); nsms.append(s.ns_ms + s.apply_ms)
    prep_ms, ns_ms = float(np.median(prep)), float(np.median(nsms))
    nominal = sum(k * ns_flops(r, c)[0] for r, c, k in tensors)
    algorithmic = sum(k * ns_flops(r, c)[1] for r, c, k in tensors)
    single_kernel = all(nsm.muon_get_bucket_info(plan, b).ns_single_kernel for b in range(info.n_buckets))
    executed = sum(k * ns_executed_flops(r, c, small=single_kernel) for r, c, k in tensors)
    # G read, M read and written, X0 written: bf16, or in 3xTF32 mode fp32 hi and lo of X0 and X0^T
    x0_bytes = 16 if tf32 else 2
    prep_bytes = sum(G[i].numel() * (G[i].element_size() + 4 + 4 + x0_bytes) for i in range(len(tensors)))
    peaks, peak_kind = load_peaks()
    bf16_sustained = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    peak_tf, peak_name = choose_bf16_peak(peaks, peak_kind, clocks, ms * 1e-3 * args.steps)
    ns_alg_tflops = algorithmic / (ns_ms * 1e-3) / 1e12
    if tf32:
        # 3xTF32: three kind::tf32 products per product, against cuBLAS's tf32 GEMM
        # timed now (after the timed region, so it does not heat the GPU for it)
        peak_tf = measure_tf32_gemm_tflops()
        peak_name = ("cuBLAS tf32 GEMM measured in this run (torch.matmul, 8192^3 fp32 with TF32 "
                     f"tensor cores, burst; half the bf16 figure would be {tf32_peak(peaks['bf16_tflops']):.1f}); "
                     "achieved counts the three tf32 products of each product")
    ns_launches = launches_per_step(nsm, plan, info, ns_only=True)
    # the single-launch kernel for m <= 128 reads X0 once and the weights once and
    # writes the weights once (A, B' and the iterations' X stay on chip or in the
    # L2 at best): when those bytes take longer at the HBM peak than the products
    # at the tensor peak, HBM is its roofline
    ns_bytes = ns_compulsory_bytes(tensors, [W[i].element_size() for i in range(len(tensors))],
                                   [G[i].element_size() for i in range(len(tensors))], momentum_fused, NS_METHOD)
    hbm_bound = single_kernel and not tf32 and hbm_binds(ns_bytes, algorithmic, peaks["hbm_gbs"], peak_tf)

    # ---- end to end through the C ABI with host buffers ----
    # Every step uploads that step's gradients from pinned host memory (on a copy
    # stream, into one of two device buffers, so step i+1's upload overlaps step i)
    # and reads back the step's result status word; a second variant reads the
    # updated weights back every step instead (no overlap possible: the next step
    # rewrites them).
    e2e = None
    if args.workload in ("layer", "single"):
        hG = [g.cpu().pin_memory() for g in G]
        dG = [G, [torch.empty_like(g) for g in G]]
        hstat = [torch.zeros(8, dtype=torch.uint8).pin_memory() for _ in range(2)]
        copy = torch.cuda.Stream()
        loaded = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        for ev in consumed:
            ev.record(stream)

        def e2e_step(i):
            b = i % 2
            with torch.cuda.stream(copy):
                copy.wait_event(consumed[b])
                for dg, hg in zip(dG[b], hG):
                    dg.copy_(hg, non_blocking=True)
                loaded[b].record(copy)
            stream.wait_event(loaded[b])
            step(dG[b])
            hstat[b].copy_(ws[:8], non_blocking=True)
            consumed[b].record(stream)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        k_e2e = max(3, min(args.steps, 100))
        e0.record(stream)
        for i in range(k_e2e):
            e2e_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / k_e2e
        hW = [torch.empty_like(w, device="cpu").pin_memory() for w in W]

        def e2e_w_step():
            for dg, hg in zip(G, hG):
                dg.copy_(hg, non_blocking=True)
            step()
            for hw, dw in zip(hW, W):
                hw.copy_(dw, non_blocking=True)

        e2e_w_step()
        torch.cuda.synchronize()
        k_w = max(3, min(args.steps, 30))
        e0.record(stream)
        for _ in range(k_w):
            e2e_w_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_w_ms = e0.elapsed_time(e1) / k_w
        e2e_ms, e2e_w_ms = max_over_ranks([e2e_ms, e2e_w_ms])
        h2d = sum(g.numel() * g.element_size() for g in hG)
        e2e = {"value": whole_job_rate(n_mats, world, e2e_ms), "unit": "matrices/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": 8, "ms_per_step": e2e_ms,
               "note": "gradients uploaded every step (overlapping the previous step); status word read back",
               "weights_readback": {"value": whole_job_rate(n_mats, world, e2e_w_ms), "unit": "matrices/s",
                                    "h2d_bytes_per_step": h2d,
                                    "d2h_bytes_per_step": sum(w.numel() * w.element_size() for w in hW),
                                    "ms_per_step": e2e_w_ms}}

    line = {
        "metric": METRIC, "value": value, "unit": "matrices/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "tf32x3" if tf32 else "bf16", "data": "synthetic",
        "config": arm_config(spec, world),
        "plan": {"buckets": int(info.n_buckets), "bucket_cap_bytes": cap, "ns_schedule_detail": schedule,
                 "momentum_in_ns_kernel": momentum_fused},
        "ns_tflops": {"nominal": nominal / (ms * 1e-3) / 1e12, "algorithmic_in_ns_phase": ns_alg_tflops,
                      "executed_in_ns_phase": executed / (ns_ms * 1e-3) / 1e12,
                      "frac_of_sustained_peak_executed": executed / (ns_ms * 1e-3) / 1e12 / bf16_sustained,
                      "frac_of_burst_peak_executed": executed / (ns_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]},
        "phase_ms": {"prep": prep_ms, "ns_and_apply": ns_ms,
                     "note": "the weight update runs in the last UPDATE GEMM's epilogue"},
        "elementwise_gbs": ({"prep": None, "peak": peaks["hbm_gbs"], "prep_frac": None,
                             "note": "the momentum runs inside the small-matrix Newton-Schulz kernel; its bytes "
                                     "are in the roofline's compulsory bytes"} if momentum_fused else
                            {"prep": prep_bytes / (prep_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                             "prep_frac": prep_bytes / (prep_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}),
        "roofline": roofline_entry(nsm, plan, info, tf32, hbm_bound, ns_ms, ns_launches, algorithmic, executed,
                                   ns_bytes, peak_tf, peak_name, peaks, bf16_sustained,
                                   ns_gemm_traffic() if args.workload == "layer" and not tf32 else
                                   head_traffic(NS_METHOD, n_mats) if args.workload == "heads" and not momentum_fused
                                   and NS_STEPS == 5 else None,
                                   ("algorithmic bytes: " + ("G read, M read and written" if momentum_fused
                                                             else "X0 read") +
                                    (", X0 written and read back once more for U = R X0" if momentum_fused and
                                     NS_METHOD == "gram" else ", X0 read again for U = R X0"
                                     if NS_METHOD == "gram" else "") +
                                    ", weights read and written once")),
        "clocks": clocks,
        "gpu_launches": args.steps * launches_per_step(nsm, plan, info),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_library_baseline and not tf32 and NS_METHOD == "standard" and NS_SCHEDULE["kind"] == "fixed":
        k_lib = max(1, min(args.steps, 10 if args.workload != "experts" else 2))
        lib_ms = max_over_ranks([library_step_ms(torch, W, M, G, k_lib, [NS_COEFFS] * NS_STEPS)])[0]
        line["library_baseline"] = {
            "value": whole_job_rate(n_mats, world, lib_ms), "unit": "matrices/s", "ms_per_step": lib_ms,
            "steps": k_lib, "speedup_of_value": lib_ms / ms,
            "what": "the same step as a per-tensor loop of torch ops on this GPU (cuBLAS bf16 batched GEMMs "
                    "with fp32 accumulation, fp32 momentum and norm), timed after the measurements above"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_leg(args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)
    del ws
    if world > 1:
        dist.destroy_process_group()


def host_link_peaks(torch, n_bytes=2 << 30):
    """Pinned host <-> device copy bandwidth: one direction at a time, then both at once."""
    h1 = torch.empty(n_bytes, dtype=torch.uint8).pin_memory()
    h2 = torch.empty(n_bytes, dtype=torch.uint8).pin_memory()
    d1 = torch.empty(n_bytes, dtype=torch.uint8, device="cuda")
    d2 = torch.empty(n_bytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t) / reps

    def both():
        with torch.cuda.stream(s1):
            d1.copy_(h1, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)

    out = {"h2d_gbs": n_bytes / timed(lambda: d1.copy_(h1, non_blocking=True)) / 1e9,
           "d2h_gbs": n_bytes / timed(lambda: h2.copy_(d2, non_blocking=True)) / 1e9,
           "bidirectional_gbs": 2 * n_bytes / timed(both) / 1e9,
           "method": "cudaMemcpyAsync of 2 GiB pinned buffers, one direction, then both on two streams"}
    del h1, h2, d1, d2
    return out


def run_offload(args):
    """36 Qwen3-4B layers with gradients and fp32 momentum in pinned host memory."""
    import torch
    from newton_schulz_muon_gb300.build import build
    build()
    import newton_schulz_muon_gb300 as nsm
    import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    shapes = [(r, c) for _ in range(36) for _, r, c in QWEN3_4B_LAYER]
    zero_copy = args.offload_mode == "zerocopy"
    cfg = nsm.muon_config_default(offload=1, max_inflight=2, timing=1, offload_zero_copy=1 if zero_copy else 0)
    plan = nsm.muon_plan(shapes, bucket_cap_bytes=128 << 20, config=cfg)
    info = nsm.muon_get_plan_info(plan)
    ws = nsm.allocate_workspace(plan)
    schedule = set_schedule(nsm, plan)
    hG, hM, hU = [], [], []
    for i, (r, c) in enumerate(shapes):
        g = torch.empty((r, c), dtype=torch.bfloat16, device="cuda")
        mm = torch.empty((r, c), dtype=torch.float32, device="cuda")
        synth.fill_normal_cuda(g, synth.SEED, synth.stream_id(i, synth.ROLE_G), 0, G_SIGMA)
        synth.fill_normal_cuda(mm, synth.SEED, synth.stream_id(i, synth.ROLE_M), 0, M_SIGMA)
        hG.append(torch.empty((r, c), dtype=torch.bfloat16, pin_memory=True).copy_(g))
        hM.append(torch.empty((r, c), dtype=torch.float32, pin_memory=True).copy_(mm))
        hU.append(torch.empty((r, c), dtype=torch.float32, pin_memory=True))
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        nsm.muon_offload_step(plan, hG, hM, hU, MU, True, NS_STEPS)
    times, h2d, d2h = [], [], []
    sampler = ClockSampler(local)
    sampler.start()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        a = time.perf_counter()
        nsm.muon_offload_step(plan, hG, hM, hU, MU, True, NS_STEPS)
        times.append(time.perf_counter() - a)
        st = nsm.muon_get_stats(plan)
        h2d.append(st.h2d_ms); d2h.append(st.d2h_ms)
    total = time.perf_counter() - t0
    clocks = sampler.stop()
    s_ms = 1000 * float(np.median(times))
    link = host_link_peaks(torch)
    hb, db = st.h2d_bytes, st.d2h_bytes
    algorithmic = sum(ns_flops(r, c)[1] for r, c in shapes)
    line = {"metric": METRIC, "value": len(shapes) / (s_ms / 1000), "unit": "matrices/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": s_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": offload_config(world, zero_copy),
            "plan": {"buckets": int(info.n_buckets), "ns_schedule_detail": schedule},
            "host_link": {"h2d_bytes_per_step": hb, "d2h_bytes_per_step": db,
                          "h2d_gbs_avg_over_step": hb / (s_ms * 1e-3) / 1e9,
                          "d2h_gbs_avg_over_step": db / (s_ms * 1e-3) / 1e9,
                          "h2d_copy_ms_sum": float(np.median(h2d)), "d2h_copy_ms_sum": float(np.median(d2h)),
                          "h2d_gbs_while_copying": hb / (float(np.median(h2d)) * 1e-3) / 1e9,
                          "d2h_gbs_while_copying": db / (float(np.median(d2h)) * 1e-3) / 1e9,
                          "measured_link": link,
                          "step_floor_ms": 1000 * max(db / (link["d2h_gbs"] * 1e9), hb / (link["h2d_gbs"] * 1e9),
                                                      (hb + db) / (link["bidirectional_gbs"] * 1e9)),
                          "frac_of_link_floor": 1000 * max(db / (link["d2h_gbs"] * 1e9),
                                                           hb / (link["h2d_gbs"] * 1e9),
                                                           (hb + db) / (link["bidirectional_gbs"] * 1e9)) / s_ms},
            "ms_per_step_best": 1000 * float(np.min(times)),
            "ns_tflops_algorithmic_over_step": algorithmic / (s_ms * 1e-3) / 1e12,
            "wall_s": total, "clocks": clocks,
            "gpu_launches": args.steps * launches_per_step(nsm, plan, info)}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_leg("offload")
    print(json.dumps(line), flush=True)
    del ws


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-library-baseline", action="store_true",
                    help="skip timing the same step as a loop of torch (cuBLAS) ops on the GPU")
    ap.add_argument("--workload", choices=["layer", "single", "heads", "experts", "offload"], default="layer",
                    help="layer (default, the headline) or another measured workload")
    ap.add_argument("--ns-precision", choices=["bf16", "tf32x3"], default="bf16",
                    help="Newton-Schulz arithmetic: bf16 (default) or the 3xTF32 accuracy mode")
    ap.add_argument("--layers", type=int, default=None,
                    help="heads / experts: fewer layers than the full workload (profiling captures)")
    ap.add_argument("--bucket-cap-mib", type=int, default=None,
                    help="micro-bucket cap in MiB of wide-form bf16 matrix bytes (default: the workload's own)")
    ap.add_argument("--ns-method", choices=["standard", "gram"], default="standard",
                    help="Newton-Schulz on X (standard) or on X X^T (gram: small-matrix buckets only, X read twice)")
    ap.add_argument("--momentum", choices=["separate", "fused"], default="separate",
                    help="small-matrix buckets: the momentum kernel first (default, the library's default), or "
                         "the momentum computed in the Newton-Schulz kernel's first pass")
    ap.add_argument("--offload-mode", choices=["copy", "zerocopy"], default="copy",
                    help="offload workload: staged copies (default) or zero-copy kernel access to host memory")
    ap.add_argument("--ns-steps", type=int, default=5, help="Newton-Schulz iterations per step (default 5)")
    ap.add_argument("--ns-schedule", choices=["fixed", "minimax"], default="fixed",
                    help="fixed (3.4445, -4.7750, 2.0315) every iteration, or the per-iteration minimax schedule")
    ap.add_argument("--ns-lower", type=float, default=1e-3, help="minimax: assumed lower end of the singular values")
    ap.add_argument("--ns-safety", type=float, default=1.05, help="minimax: widening of each fitted interval's top")
    args = ap.parse_args()
    global NS_STEPS, NS_METHOD
    NS_STEPS = args.ns_steps
    NS_METHOD = args.ns_method
    NS_SCHEDULE.update(kind=args.ns_schedule, lower=args.ns_lower, safety=args.ns_safety)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "offload":
        run_offload(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
