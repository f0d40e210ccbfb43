#!/usr/bin/env python
"""Benchmark of the hot path on one GB300 (or N replicas under torchrun).

One step = one pass of the whole path over one batch of synthetic inputs:
  1. persistent all-gather: W=8 logical ranks, 4096 x 4096 f16 per rank
     (uniform[-1,1]), explicit tile 8x256, 148 programs, local copy first
     then peers rotated;
  2. fused matmul + all-gather: W=8, M_local=1024, N=3584, K=8192, f16 in,
     f32 accumulate, f16 out, 128x256 tcgen05 tiles, inputs normal(0,1)/sqrt(K).
Every rank's 8 logical ranks live in one symmetric heap on its own GPU; the
per-step working set (about 3 GB) is far larger than L2.

The metric is the step's roofline time (gather bytes at the measured HBM
peak + fused FLOPs at the measured dense f16 tensor peak) as a percentage of
the measured step time; the absolute GB/s and TFLOP/s of each kernel are in
the same line.  ``--impl reference`` times the CPU oracle on a bounded
sample of the same step instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "all-gather HBM GB/s & fused GEMM+gather TFLOP/s, % of roofline, 1xGB300"
UNIT = "% of roofline"

GATHER = dict(W=8, M=4096, N=4096, es=2, tile=(8, 256), programs=148)
FUSED = dict(W=8, M=1024, N=3584, K=8192, tile=(128, 256))

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
F16_PER_BF16 = 1.0  # nominal dense f16 : bf16 tensor rate


def gather_bytes(c=GATHER) -> float:
    """Algorithmic bytes: every rank's block read once, W copies of W blocks written."""
    blk = c["M"] * c["N"] * c["es"]
    return c["W"] * blk + c["W"] * c["W"] * blk


def fused_flops(c=FUSED) -> float:
    return 2.0 * c["W"] * c["M"] * c["N"] * c["K"]


def fused_bytes(c=FUSED) -> float:
    """A of every rank + B once + W copies of every rank's C block."""
    return 2.0 * (c["W"] * c["M"] * c["K"] + c["K"] * c["N"] + c["W"] ** 2 * c["M"] * c["N"])


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def roofline_times(peaks):
    hbm = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12 * F16_PER_BF16
    t_g = gather_bytes() / hbm
    t_f = max(fused_flops() / tc, fused_bytes() / hbm)
    return t_g, t_f


def source_sha(name: str) -> str:
    with open(os.path.join(ROOT, "gemm_gather_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_for(kernel: str, src: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or
    None when the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f).get(kernel)
    if not t or t.get("source_sha") != source_sha(src):
        return None
    return t.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, out_path: str | None):
        self.index = index
        self.out_path = out_path
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.strip()]
        if self.out_path:
            with open(self.out_path, "w") as f:
                f.write(self.QUERY + "\n" + out)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip() == "Active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- #
# CPU oracle on a bounded sample (reference arm and cpu_baseline)             #
# --------------------------------------------------------------------------- #

def oracle_sample_step(orc, gather_rows: int, fused_rows: int, seed: int = 0):
    """One sampled step of the oracle: the gather on `gather_rows` of the
    4096 rows per rank, the fused path on `fused_rows` of the 1024 rows per
    rank (all N columns, full K).  Returns (gather seconds, fused seconds)."""
    import numpy as np
    import torch

    import gg_inputs
    g, f = GATHER, FUSED
    W = g["W"]
    gen = gg_inputs.generator(seed)
    # gather sample heap: input block + gathered output per partition
    blk = gather_rows * g["N"] * 2
    part = blk + W * blk
    heap = np.full(W * part, gg_inputs.SENTINEL_BYTE, dtype=np.uint8)
    for h in range(W):
        x = gg_inputs.uniform_pm1((gather_rows, g["N"]), torch.float16, gen)
        heap[h * part: h * part + blk] = x.view(torch.int16).numpy().view(np.uint8).ravel()
    # fused sample heap: A rows + gathered output per partition
    a_bytes = fused_rows * f["K"] * 2
    c_bytes = W * fused_rows * f["N"] * 2
    fpart = a_bytes + c_bytes
    fheap = np.zeros(W * fpart, dtype=np.uint8)
    for h in range(W):
        a = gg_inputs.normal((fused_rows, f["K"]), torch.float16, gen, scale=f["K"] ** -0.5)
        fheap[h * fpart: h * fpart + a_bytes] = a.view(torch.int16).numpy().view(np.uint8).ravel()
    B = gg_inputs.normal((f["K"], f["N"]), torch.float16, gen, scale=f["K"] ** -0.5)
    Bb = B.view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    orc.all_gather(heap, part, 0, g["N"], blk, g["N"], gather_rows, g["N"], 2, (0, 1, W))
    t1 = time.perf_counter()
    orc.matmul_all_gather(fheap, fpart, 0, f["K"], Bb, a_bytes, f["N"], fused_rows, f["N"],
                          f["K"], 0, (0, 1, W))
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def size_sample(orc, seconds: float):
    """Rows of the gather and of the fused path whose oracle run takes about
    `seconds` (30% gather, 70% fused), from a small calibration run."""
    cg, cf = 16, 4
    t_g, t_f = oracle_sample_step(orc, cg, cf)
    rows_g = int(max(8, min(GATHER["M"], cg * 0.3 * seconds / max(t_g, 1e-6))))
    rows_f = int(max(1, min(FUSED["M"], cf * 0.7 * seconds / max(t_f, 1e-6))))
    return rows_g, rows_f


def cpu_baseline(peaks, budget_s: float = 15.0):
    import oracle
    orc = oracle.Oracle()
    cores = orc.max_threads()
    t_rg, t_rf = roofline_times(peaks)
    rows_g, rows_f = size_sample(orc, budget_s)
    t_g, t_f = oracle_sample_step(orc, rows_g, rows_f)
    t_full = t_g * GATHER["M"] / rows_g + t_f * FUSED["M"] / rows_f
    value = 100.0 * (t_rg + t_rf) / t_full
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"gather on {rows_g} of 4096 rows per rank ({t_g:.2f} s) and fused path "
                       f"on {rows_f} of 1024 rows per rank, full K and N ({t_f:.2f} s); "
                       f"scaled by rows to a full step: {t_full:.1f} s/step"),
            "seconds_per_step": t_full}


# --------------------------------------------------------------------------- #
# reference arm                                                               #
# --------------------------------------------------------------------------- #

def run_reference(args, peaks, peak_src):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    orc = oracle.Oracle()
    cores = orc.max_threads()
    t_rg, t_rf = roofline_times(peaks)
    # size each step's sample so warmup + steps finish in about two minutes
    rows_g, rows_f = size_sample(orc, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_step(orc, rows_g, rows_f)
    total = 0.0
    for _ in range(args.steps):
        t_g, t_f = oracle_sample_step(orc, rows_g, rows_f)
        total += t_g + t_f
    # the sampled step holds this share of the full step's roofline time
    sample_roof = t_rg * (rows_g / GATHER["M"]) + t_rf * (rows_f / FUSED["M"])
    value = 100.0 * sample_roof / (total / args.steps)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": config_block(peaks, peak_src),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": (f"each step: oracle gather on {rows_g} of 4096 rows per rank "
                                    f"and fused path on {rows_f} of 1024 rows per rank")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_block(peaks, peak_src):
    return {
        "workload": ("all_gather W=8 4096x4096 f16 tile 8x256 148 programs + "
                     "matmul_all_gather W=8 M_local=1024 N=3584 K=8192 f16 tile 128x256"),
        "all_gather": {"W": 8, "M_local": 4096, "N": 4096, "dtype": "f16", "tile": [8, 256],
                       "comm_programs": GATHER["programs"], "values": "uniform[-1,1]"},
        "matmul_all_gather": {"W": 8, "M_local": 1024, "N": 3584, "K": 8192, "dtype": "f16",
                              "tile": [128, 256], "values": "normal(0,1)/sqrt(K)"},
        "l2": "inputs larger than L2 (about 3 GB touched per step)",
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "f16_tflops": peaks["bf16_tflops"] * F16_PER_BF16,
                  "source": peak_src,
                  "note": "f16 dense peak = measured bf16 burst peak x nominal 1:1 ratio"},
        "seed": 0,
    }


# --------------------------------------------------------------------------- #
# the GPU arm                                                                 #
# --------------------------------------------------------------------------- #

def setup_device(dev, seed=0):
    import torch

    import gemm_gather_gb300 as gg
    import gg_inputs
    g, f = GATHER, FUSED
    W = g["W"]
    gin = g["M"] * g["N"] * 2
    gout = W * gin
    fa = f["M"] * f["K"] * 2
    fout = W * f["M"] * f["N"] * 2
    align = 1 << 16
    offs = {}
    o = 0
    for name, size in (("g_in", gin), ("g_out", gout), ("f_a", fa), ("f_out", fout)):
        offs[name] = o
        o += (size + align - 1) // align * align
    part = o
    sh = gg.SymmetricHeap(W, part, device=dev)
    gen = gg_inputs.generator(seed)
    host = {"g_in": [], "f_a": []}
    for h in range(W):
        x = gg_inputs.uniform_pm1((g["M"], g["N"]), torch.float16, gen)
        host["g_in"].append(x)
        sh.view(h, offs["g_in"], g["M"], g["N"], g["N"], torch.float16).copy_(x.to(dev))
    for h in range(W):
        a = gg_inputs.normal((f["M"], f["K"]), torch.float16, gen, scale=f["K"] ** -0.5)
        host["f_a"].append(a)
        sh.view(h, offs["f_a"], f["M"], f["K"], f["K"], torch.float16).copy_(a.to(dev))
    B = gg_inputs.normal((f["K"], f["N"]), torch.float16, gen, scale=f["K"] ** -0.5)
    host["B"] = B
    Bd = B.to(dev)
    torch.cuda.synchronize(dev)
    return sh, offs, Bd, host


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gather-path", default="auto", choices=["auto", "bulk", "vector"])
    ap.add_argument("--fused-programs", type=int, default=0, help="0: one CTA per SM")
    ap.add_argument("--clocks-out", default=None)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    peaks, peak_src = load_peaks()
    if args.impl == "reference":
        return run_reference(args, peaks, peak_src)

    import torch
    import torch.distributed as dist

    import gemm_gather_gb300 as gg

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fused_programs = args.fused_programs or sms
    g, f = GATHER, FUSED
    W = g["W"]
    group = (0, 1, W)
    sh, offs, Bd, host = setup_device(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        gg.all_gather(sh.heap, -1, sh.ptr(0, offs["g_in"]), g["N"], sh.ptr(0, offs["g_out"]),
                      g["N"], g["M"], g["N"], torch.float16, g["tile"], g["programs"], group,
                      status=status, stream=stream, path=args.gather_path)
        if ev is not None:
            ev[1].record(stream)
        gg.matmul_all_gather(sh.heap, -1, sh.ptr(0, offs["f_a"]), f["K"], Bd, f["N"],
                             sh.ptr(0, offs["f_out"]), f["N"], f["M"], f["N"], f["K"],
                             torch.float16, f["tile"], fused_programs, group, status=status,
                             stream=stream)
        if ev is not None:
            ev[2].record(stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local, args.clocks_out) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if clocks:
        clocks.mark(True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    barrier()
    if clocks:
        clocks.mark(False)
    clk = clocks.stop() if clocks else None
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the timed steps")
    elapsed_ms = t_start.elapsed_time(t_end)
    g_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    f_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    ms_step = elapsed_ms / args.steps

    # ---- end to end through the C ABI, host buffers, copies in the timed region
    pinned_in = [x.pin_memory() for x in host["g_in"]]
    pinned_a = [x.pin_memory() for x in host["f_a"]]
    pinned_b = host["B"].pin_memory()
    out_g = torch.empty((W, W * g["M"], g["N"]), dtype=torch.float16).pin_memory()
    out_f = torch.empty((W, W * f["M"], f["N"]), dtype=torch.float16).pin_memory()
    h2d = sum(x.numel() * 2 for x in pinned_in) + sum(x.numel() * 2 for x in pinned_a) \
        + pinned_b.numel() * 2
    d2h = out_g.numel() * 2 + out_f.numel() * 2

    def e2e_step():
        for h in range(W):
            sh.view(h, offs["g_in"], g["M"], g["N"], g["N"], torch.float16).copy_(
                pinned_in[h], non_blocking=True)
            sh.view(h, offs["f_a"], f["M"], f["K"], f["K"], torch.float16).copy_(
                pinned_a[h], non_blocking=True)
        Bd.copy_(pinned_b, non_blocking=True)
        step()
        for h in range(W):
            out_g[h].copy_(sh.view(h, offs["g_out"], W * g["M"], g["N"], g["N"], torch.float16),
                           non_blocking=True)
            out_f[h].copy_(sh.view(h, offs["f_out"], W * f["M"], f["N"], f["N"], torch.float16),
                           non_blocking=True)

    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    for _ in range(3):
        e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    # ---- roofline bookkeeping
    t_rg, t_rf = roofline_times(peaks)
    roof_step = t_rg + t_rf
    value = 100.0 * world * roof_step / (ms_step * 1e-3)
    e2e_value = 100.0 * world * roof_step / (e2e_ms * 1e-3)
    g_gbs = gather_bytes() / (g_ms * 1e-3) / 1e9
    f_tfs = fused_flops() / (f_ms * 1e-3) / 1e12
    hbm_peak = peaks["hbm_gbs"]
    tc_peak = peaks["bf16_tflops"] * F16_PER_BF16
    kernels = {
        "all_gather": {"kernel": "ag_bulk_kernel" if args.gather_path != "vector" else "ag_vec_kernel",
                       "ms": g_ms, "GB/s": g_gbs, "roofline_ms": 1e3 * t_rg,
                       "frac": g_gbs / hbm_peak, "bound": "hbm",
                       "algorithmic_bytes": gather_bytes()},
        "matmul_all_gather": {"kernel": "mag_kernel", "ms": f_ms, "TFLOP/s": f_tfs,
                              "roofline_ms": 1e3 * t_rf, "frac": f_tfs / tc_peak,
                              "bound": "tensor", "algorithmic_flops": fused_flops(),
                              "programs": fused_programs},
    }
    if g_ms >= f_ms:
        roof = {"kernel": "ag_bulk_kernel", "bound": "hbm", "achieved": g_gbs, "peak": hbm_peak,
                "unit": "GB/s", "frac": g_gbs / hbm_peak,
                "traffic": traffic_for("ag_bulk_kernel", "ag_kernels.cu"),
                "per_unit": "bytes = W*M*N*s reads + W^2*M*N*s writes per launch"}
    else:
        roof = {"kernel": "mag_kernel", "bound": "tensor", "achieved": f_tfs, "peak": tc_peak,
                "unit": "TFLOP/s", "frac": f_tfs / tc_peak,
                "traffic": traffic_for("mag_kernel", "mag_kernel.cu"),
                "per_unit": "FLOPs = 2*W*M*N*K per launch"}
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else peak_src
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    cpu = None if args.no_cpu_baseline else cpu_baseline(peaks)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": config_block(peaks, peak_src),
        "kernels": kernels,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "path": "pinned host -> heap (cudaMemcpyAsync) -> C-ABI calls -> pinned host"},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "device": torch.cuda.get_device_name(dev), "sms": sms,
        "torch": torch.__version__,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
