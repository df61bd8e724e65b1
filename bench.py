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
G_SIGMA, W_SIGMA, M_SIGMA = 1e-3, 0.02, 0.02


def ns_flops(rows, cols, steps=NS_STEPS):
    """(nominal, algorithmic) Newton-Schulz flops of one rows x cols matrix."""
    m, n = min(rows, cols), max(rows, cols)
    nominal = steps * (4 * m * m * n + 2 * m ** 3)
    algorithmic = steps * (m * (m + 1) * n + 2 * m ** 3 + 2 * m * m * n)
    return nominal, algorithmic


def ns_executed_flops(rows, cols, steps=NS_STEPS, bm=128, bn=256, bk=64):
    """Flops the tensor cores execute: whole 128x256 tiles, k rounded up to 64."""
    m, n = min(rows, cols), max(rows, cols)
    cd = lambda a, b: -(-a // b)
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


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# CPU oracle timing (bench's cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_inputs(names):
    import synth
    out = {}
    for i, (name, r, c) in enumerate(QWEN3_4B_LAYER):
        if name not in names:
            continue
        W = synth.tensor(synth.SEED, synth.stream_id(i, synth.ROLE_W), 0, (r, c), W_SIGMA, synth.F32)
        M = synth.tensor(synth.SEED, synth.stream_id(i, synth.ROLE_M), 0, (r, c), M_SIGMA, synth.F32)
        G = synth.tensor(synth.SEED, synth.stream_id(i, synth.ROLE_G), 0, (r, c), G_SIGMA, synth.BF16)
        out[name] = (W.astype(np.float64), M, synth.as_f64(G, synth.BF16))
    return out


def oracle_step(inputs, names):
    import oracle
    for name in names:
        W, M, G = inputs[name]
        oracle.muon_matrix_step(W, M, G, LR, MU, True, WD, NS_STEPS)


def cpu_baseline_leg():
    names = [n for n, _, _ in QWEN3_4B_LAYER]
    inputs = oracle_inputs(names)
    t0 = time.perf_counter()
    oracle_step(inputs, names)
    dt = time.perf_counter() - t0
    return {"value": len(names) / dt, "unit": "matrices/s", "cores": cores_used(), "kind": "oracle",
            "sample": f"one full step of the 7-matrix layer ({dt:.1f} s, numpy fp64, OpenBLAS threads)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    names_all = [n for n, _, _ in QWEN3_4B_LAYER]
    inputs = oracle_inputs(names_all)
    for _ in range(args.warmup):            # warm-up on the smallest matrix only
        oracle_step(inputs, ["k_proj"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(inputs, names_all)
    dt = time.perf_counter() - t0
    value = args.steps * len(names_all) / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "matrices/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "matrices_per_step": 7},
        "cpu_baseline": {"value": value, "unit": "matrices/s", "cores": cores_used(), "kind": "oracle",
                         "sample": "each timed step is one full oracle step of the 7-matrix layer; "
                                   "warm-up steps run k_proj only"},
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
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


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

    shapes = [(r, c, 1, 0) for _, r, c in QWEN3_4B_LAYER]
    cfg = nsm.muon_config_default(timing=1)
    plan = nsm.muon_plan(shapes, bucket_cap_bytes=512 << 20, config=cfg)
    info = nsm.muon_get_plan_info(plan)
    ws = nsm.allocate_workspace(plan)
    W, M, G = [], [], []
    for i, (_, r, c) in enumerate(QWEN3_4B_LAYER):
        w = torch.empty((r, c), dtype=torch.float32, device="cuda")
        mm = torch.empty((r, c), dtype=torch.float32, device="cuda")
        g = torch.empty((r, c), dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_cuda(w, synth.SEED, synth.stream_id(i, synth.ROLE_W), 0, W_SIGMA)
        synth.fill_normal_cuda(mm, synth.SEED, synth.stream_id(i, synth.ROLE_M), 0, M_SIGMA)
        synth.fill_normal_cuda(g, synth.SEED, synth.stream_id(i, synth.ROLE_G), 0, G_SIGMA)
        W.append(w); M.append(mm); G.append(g)
    stream = torch.cuda.current_stream()

    def step():
        nsm.muon_step(plan, W, G, M, LR, MU, True, WD, NS_STEPS, stream)

    for _ in range(args.warmup):
        step()
    st, nf = nsm.muon_sync(plan, stream)
    if st != nsm.MUON_OK:
        raise RuntimeError(f"device status {st} after warm-up")

    # ---- timed region: K steps, inputs (1.0 GB) larger than L2 ----
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
    if world > 1:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    st, nf = nsm.muon_sync(plan, stream)
    if st != nsm.MUON_OK:
        raise RuntimeError(f"device status {st} after the timed region")
    n_mats = len(QWEN3_4B_LAYER)
    value = n_mats * world / (ms / 1000.0)

    # ---- per-phase times (CUDA events inside the library, one step at a time) ----
    prep, nsms = [], []
    for _ in range(5):
        step()
        s = nsm.muon_get_stats(plan)
        prep.append(s.prep_ms); nsms.append(s.ns_ms + s.apply_ms)
    prep_ms, ns_ms = float(np.median(prep)), float(np.median(nsms))
    nominal = sum(ns_flops(r, c)[0] for _, r, c in QWEN3_4B_LAYER)
    algorithmic = sum(ns_flops(r, c)[1] for _, r, c in QWEN3_4B_LAYER)
    executed = sum(ns_executed_flops(r, c) for _, r, c in QWEN3_4B_LAYER)
    elems = sum(r * c for _, r, c in QWEN3_4B_LAYER)
    prep_bytes = 12 * elems
    peaks, peak_kind = load_peaks()
    peak_tf = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    ns_alg_tflops = algorithmic / (ns_ms * 1e-3) / 1e12
    ns_launches = 3 * NS_STEPS * info.n_buckets

    # ---- end to end through the C ABI with host buffers ----
    hG = [g.cpu().pin_memory() for g in G]
    hW = [torch.empty_like(w, device="cpu").pin_memory() for w in W]
    h2d = sum(g.numel() * g.element_size() for g in hG)
    d2h = sum(w.numel() * w.element_size() for w in hW)

    def e2e_step():
        for dg, hg in zip(G, hG):
            dg.copy_(hg, non_blocking=True)
        step()
        for hw, dw in zip(hW, W):
            hw.copy_(dw, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    k_e2e = max(3, min(args.steps, 50))
    e0.record(stream)
    for _ in range(k_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / k_e2e
    if world > 1:
        t = torch.tensor([e2e_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    line = {
        "metric": METRIC, "value": value, "unit": "matrices/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "matrices_per_step": n_mats, "elements_per_step": elems,
                   "buckets": int(info.n_buckets), "parallelism": f"replicas{world}",
                   "l2": "inputs 1.0 GB per step, larger than the 129 MB L2"},
        "ns_tflops": {"nominal": nominal / (ms * 1e-3) / 1e12, "algorithmic_in_ns_phase": ns_alg_tflops,
                      "executed_in_ns_phase": executed / (ns_ms * 1e-3) / 1e12,
                      "frac_of_sustained_peak_executed": executed / (ns_ms * 1e-3) / 1e12 / peak_tf,
                      "frac_of_burst_peak_executed": executed / (ns_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]},
        "phase_ms": {"prep": prep_ms, "ns_and_apply": ns_ms,
                     "note": "the weight update runs in the last UPDATE GEMM's epilogue"},
        "elementwise_gbs": {"prep": prep_bytes / (prep_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                            "prep_frac": prep_bytes / (prep_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "roofline": {"bound": "tensor", "kernel": "ns_gemm_kernel (bf16, with the fused weight update)",
                     "achieved": ns_alg_tflops, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": ns_alg_tflops / peak_tf, "traffic": None,
                     "peak_kind": f"{peak_kind} bf16 sustained (kernel runs inside multi-second loops)",
                     "per_launch_ms": ns_ms / ns_launches,
                     "algorithmic_flops_per_launch": algorithmic / ns_launches},
        "clocks": clocks,
        "e2e": {"value": n_mats * world / (e2e_ms / 1000.0), "unit": "matrices/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * info.n_buckets * (2 + 3 * NS_STEPS),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_leg()
    if rank == 0:
        print(json.dumps(line), flush=True)
    del ws
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
