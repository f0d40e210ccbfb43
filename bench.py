#!/usr/bin/env python
"""Benchmark of the hot path on one GB300 (or N replicas under torchrun).

One step = one pass of the whole path over one batch of synthetic inputs, at
the largest configurations of the workload (the default, ``--preset largest``):
  1. persistent all-gather: W=8 logical ranks, 16384 x 8192 f32 per rank
     (normal(0,1)), explicit tile 8x256, 148 programs, local copy first then
     peers rotated (tensor-map path, runs of tiles claimed per program);
  2. fused matmul + all-gather: W=8, M_local=16384, N=3584, K=8192, f16 in,
     f32 accumulate, f16 out, 128x512 output tiles per CTA (two 128x256
     tcgen05 MMA tiles sharing each A stage; 256x512 per CTA pair),
     inputs normal(0,1)/sqrt(K).
``--preset small`` runs the smaller step instead: the W=8 4096 x 4096 f16
all-gather (uniform[-1,1]) and the fused product at M_local=1024.  Every
rank's 8 logical ranks live in one symmetric heap on its own GPU; the
per-step working set (about 48 GB; 3 GB for the small step) is far larger
than L2.

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
import os
import statistics
import subprocess
import sys
import time
from dataclasses import dataclass, replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "all-gather HBM GB/s & fused GEMM+gather TFLOP/s, % of roofline, 1xGB300"
UNIT = "% of roofline"

@dataclass
class GatherCfg:
    W: int = 8
    M: int = 4096
    N: int = 4096
    dtype: str = "f16"
    bm: int = 8
    bn: int = 256
    programs: int = 148
    start: int = 0
    stride: int = 1
    values: str = "uniform"  # uniform[-1,1] or normal(0,1)
    path: str = "auto"  # auto / tma / bulk / vector
    kind: str = "all_gather"  # all_gather / partitioned / all_to_all / ranks (W single-rank calls)
    dests_per_wait: int = 0   # destination grouping (0: all destinations at once)

    @property
    def es(self) -> int:
        return ES[self.dtype]

    def members(self):
        return [self.start + i * self.stride for i in range(self.W)]

    def describe(self) -> str:
        grp = "" if (self.start, self.stride) == (0, 1) else \
            f" group(start={self.start},stride={self.stride})"
        kern = "" if self.path == "auto" else f" {self.path}"
        grouping = f" {self.dests_per_wait} dests/wait" if self.dests_per_wait else ""
        return (f"{self.kind} W={self.W} {self.M}x{self.N} {self.dtype} tile {self.bm}x{self.bn} "
                f"{self.programs} programs{grp}{grouping}{kern}")


@dataclass
class FusedCfg:
    W: int = 8
    M: int = 1024
    N: int = 3584
    K: int = 8192
    dtype: str = "f16"
    programs: int = 0  # 0: one CTA per SM
    start: int = 0
    stride: int = 1
    path: str = "auto"  # auto / 1sm / 2sm
    bm: int = 128       # the output tile of one CTA: 128 x 512 (two MMA tiles sharing A,
    bn: int = 512       # on CTA pairs) or 128 x 256

    def members(self):
        return [self.start + i * self.stride for i in range(self.W)]

    def describe(self) -> str:
        grp = "" if (self.start, self.stride) == (0, 1) else \
            f" group(start={self.start},stride={self.stride})"
        kern = "" if self.path == "auto" else f" {self.path}"
        return (f"matmul_all_gather W={self.W} M_local={self.M} N={self.N} K={self.K} "
                f"{self.dtype} tile {self.bm}x{self.bn}{grp}{kern}")

    @property
    def tile(self):
        return (self.bm, self.bn)


ES = {"f16": 2, "bf16": 2, "f32": 4}
L2_BYTES = 126 << 20  # GB300 L2
# The benchmark's all-gathers take the library's automatic choice: the
# tensor-map path, which at 148 programs claims runs of tiles from the heap's
# workspace (load balancing across SMs).
GATHER = GatherCfg()                 # W=8 4096x4096 f16: the budget / variant sweeps' base
FUSED = FusedCfg()                   # W=8 M_local=1024
GATHER_LARGEST = GatherCfg(M=16384, N=8192, dtype="f32", values="normal")
FUSED_LARGEST = FusedCfg(M=16384)
PRESETS = {"largest": (GATHER_LARGEST, FUSED_LARGEST), "small": (GATHER, FUSED)}

# The end-to-end variant that reads every member's copy of the outputs back
# runs only while those copies fit this much pinned host memory.
E2E_ALL_COPIES_MAX_BYTES = 8 << 30

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
F16_PER_BF16 = 1.0  # nominal dense f16 : bf16 tensor rate


def parse_cfg(text: str, base):
    """'W=8,M=4096,tile=8x256,group=1:2,...' -> a copy of `base` with those fields."""
    cfg = replace(base)
    for item in filter(None, text.split(",")):
        k, v = item.split("=")
        if k == "tile":
            cfg.bm, cfg.bn = (int(x) for x in v.split("x"))
        elif k == "group":
            cfg.start, cfg.stride = (int(x) for x in v.split(":"))
        elif k in ("dtype", "values", "path", "kind"):
            setattr(cfg, k, v)
        else:
            setattr(cfg, k, int(v))
    return cfg


def gather_bytes(c: GatherCfg) -> float:
    """Algorithmic bytes: all-gather (and its partitioned form): every rank's
    block read once, W copies of W blocks written; all-to-all: each of the
    W x W blocks read once and written once."""
    blk = c.M * c.N * c.es
    if c.kind == "all_to_all":
        return 2.0 * c.W * c.W * blk
    return c.W * blk + c.W * c.W * blk


def fused_flops(c: FusedCfg) -> float:
    return 2.0 * c.W * c.M * c.N * c.K


def fused_bytes(c: FusedCfg) -> float:
    """A of every rank + B once + W copies of every rank's C block."""
    return 2.0 * (c.W * c.M * c.K + c.K * c.N + c.W ** 2 * c.M * c.N)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def roofline_times(peaks, g: GatherCfg | None, f: FusedCfg | None):
    hbm = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12 * F16_PER_BF16
    t_g = gather_bytes(g) / hbm if g else 0.0
    t_f = max(fused_flops(f) / tc, fused_bytes(f) / hbm) if f else 0.0
    return t_g, t_f


def source_sha(name: str) -> str:
    with open(os.path.join(ROOT, "gemm_gather_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# Dense f16/bf16 tensor-core FLOPs per SM per cycle (tcgen05, nominal).
TC_FLOP_PER_SM_CYCLE = 8192


def kernel_clock(rec):
    """The SM clock a traced launch ran at (gg_trace_read), or None if no
    traced launch wrote the record."""
    if not rec or not rec.get("sm_mhz"):
        return None
    return {"sm_mhz": rec["sm_mhz"], "cycles": rec["cycles"], "ns": rec["ns"],
            "source": "the launch's first CTA: clock64 and %globaltimer at its start and end"}


def traffic_for(kernel: str, src: str, workload: str):
    """Per-launch DRAM bytes of `kernel` on `workload` from the committed ncu
    summary, or None when no entry covers that workload or the kernel source
    changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entries = json.load(f).get(kernel) or []
    for t in entries if isinstance(entries, list) else [entries]:
        if t.get("bench_workload") == workload and t.get("source_sha") == source_sha(src):
            return t.get("bytes_per_launch")
    return None


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

def oracle_sample_step(orc, g: GatherCfg | None, f: FusedCfg | None, gather_rows: int,
                       fused_rows: int, seed: int = 0):
    """One sampled step of the oracle: the gather on `gather_rows` of the M
    rows per rank, the fused path on `fused_rows` of the M rows per rank (all
    N columns, full K).  Returns (gather seconds, fused seconds)."""
    import numpy as np
    import torch

    import gg_inputs
    gen = gg_inputs.generator(seed)
    t_g = t_f = 0.0
    if g is not None:
        W, es = g.W, g.es
        dt = gg_inputs.DTYPES[g.dtype]
        blk = gather_rows * g.N * es
        part = blk + W * blk
        H = g.members()[-1] + 1
        heap = np.full(H * part, gg_inputs.SENTINEL_BYTE, dtype=np.uint8)
        for h in g.members():
            x = (gg_inputs.uniform_pm1 if g.values == "uniform" else gg_inputs.normal)(
                (gather_rows, g.N), dt, gen)
            heap[h * part: h * part + blk] = x.contiguous().view(torch.uint8).numpy().ravel()
        t0 = time.perf_counter()
        orc.all_gather(heap, part, 0, g.N, blk, g.N, gather_rows, g.N, es,
                       (g.start, g.stride, W))
        t_g = time.perf_counter() - t0
    if f is not None:
        W = f.W
        dt = gg_inputs.DTYPES[f.dtype]
        a_bytes = fused_rows * f.K * 2
        fpart = a_bytes + W * fused_rows * f.N * 2
        H = f.members()[-1] + 1
        fheap = np.zeros(H * fpart, dtype=np.uint8)
        for h in f.members():
            a = gg_inputs.normal((fused_rows, f.K), dt, gen, scale=f.K ** -0.5)
            fheap[h * fpart: h * fpart + a_bytes] = a.view(torch.uint8).numpy().ravel()
        B = gg_inputs.normal((f.K, f.N), dt, gen, scale=f.K ** -0.5)
        Bb = B.view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        orc.matmul_all_gather(fheap, fpart, 0, f.K, Bb, a_bytes, f.N, fused_rows, f.N, f.K,
                              0 if f.dtype == "f16" else 1, (f.start, f.stride, W))
        t_f = time.perf_counter() - t0
    return t_g, t_f


def size_sample(orc, g, f, seconds: float):
    """Rows of the gather and of the fused path whose oracle run takes about
    `seconds` (30% gather, 70% fused when both run), from a small calibration."""
    cg, cf = 16, 4
    t_g, t_f = oracle_sample_step(orc, g, f, cg, cf)
    share_g = 0.3 if (g and f) else 1.0
    rows_g = int(max(8, min(g.M, cg * share_g * seconds / max(t_g, 1e-6)))) if g else 0
    rows_f = int(max(1, min(f.M, cf * (1 - share_g if g else 1.0) * seconds
                            / max(t_f, 1e-6)))) if f else 0
    return rows_g, rows_f


def cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo (x86 'model name'; on Arm the
    implementer / part codes), or the platform string."""
    import platform
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return platform.processor() or platform.machine()
    for key in ("model name", "Model name"):
        for line in info.splitlines():
            if line.startswith(key):
                return line.split(":", 1)[1].strip()
    impl = [l.split(":", 1)[1].strip() for l in info.splitlines() if l.startswith("CPU implementer")]
    part = [l.split(":", 1)[1].strip() for l in info.splitlines() if l.startswith("CPU part")]
    if impl and part:
        return f"{platform.machine()} implementer {impl[0]} part {part[0]}"
    return platform.processor() or platform.machine()


def cpu_baseline(peaks, g, f, budget_s: float = 15.0):
    import oracle
    orc = oracle.Oracle()
    cores = orc.max_threads()
    t_rg, t_rf = roofline_times(peaks, g, f)
    rows_g, rows_f = size_sample(orc, g, f, budget_s)
    t_g, t_f = oracle_sample_step(orc, g, f, rows_g, rows_f)
    t_full = (t_g * g.M / rows_g if g else 0.0) + (t_f * f.M / rows_f if f else 0.0)
    value = 100.0 * (t_rg + t_rf) / t_full
    parts = []
    if g:
        parts.append(f"gather on {rows_g} of {g.M} rows per rank ({t_g:.2f} s)")
    if f:
        parts.append(f"fused path on {rows_f} of {f.M} rows per rank, full K and N ({t_f:.2f} s)")
    # one thread on a smaller sample (the same rows scaled), for the per-core rate
    orc.set_threads(1)
    r1g = max(8, rows_g // 8) if g else 0
    r1f = max(1, rows_f // 8) if f else 0
    t1g, t1f = oracle_sample_step(orc, g, f, r1g, r1f)
    orc.set_threads(cores)
    t1_full = (t1g * g.M / r1g if g else 0.0) + (t1f * f.M / r1f if f else 0.0)
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": " and ".join(parts) + f"; scaled by rows to a full step: {t_full:.1f} s/step",
            "seconds_per_step": t_full,
            "single_thread": {"seconds_per_step": t1_full,
                              "sample": f"gather {r1g} rows, fused {r1f} rows per rank, scaled"},
            "cpu": cpu_model(), "nproc": os.cpu_count()}


# --------------------------------------------------------------------------- #
# reference arm                                                               #
# --------------------------------------------------------------------------- #

def run_reference(args, peaks, peak_src, g, f):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    orc = oracle.Oracle()
    cores = orc.max_threads()
    t_rg, t_rf = roofline_times(peaks, g, f)
    # size each step's sample so warmup + steps finish in about two minutes
    rows_g, rows_f = size_sample(orc, g, f, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_step(orc, g, f, rows_g, rows_f)
    total = 0.0
    for _ in range(args.steps):
        t_g, t_f = oracle_sample_step(orc, g, f, rows_g, rows_f)
        total += t_g + t_f
    # the sampled step holds this share of the full step's roofline time
    sample_roof = (t_rg * rows_g / g.M if g else 0.0) + (t_rf * rows_f / f.M if f else 0.0)
    value = 100.0 * sample_roof / (total / args.steps)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "+".join(sorted({c.dtype for c in (g, f) if c is not None})),
        "data": "synthetic", "config": config_block(peaks, peak_src, g, f),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": (f"each step: oracle gather on {rows_g} rows per rank and "
                                    f"fused path on {rows_f} rows per rank")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_block(peaks, peak_src, g, f):
    work = " + ".join(c.describe() for c in (g, f) if c is not None)
    touched = (gather_bytes(g) if g else 0) + (fused_bytes(f) if f else 0)
    cfg = {"workload": work}
    if g:
        cfg["all_gather"] = {"W": g.W, "M_local": g.M, "N": g.N, "dtype": g.dtype,
                             "tile": [g.bm, g.bn], "comm_programs": g.programs,
                             "group": [g.start, g.stride, g.W], "path": g.path,
                             "values": "uniform[-1,1]" if g.values == "uniform" else "normal(0,1)"}
    if f:
        cfg["matmul_all_gather"] = {"W": f.W, "M_local": f.M, "N": f.N, "K": f.K,
                                    "dtype": f.dtype, "tile": [f.bm, f.bn],
                                    "group": [f.start, f.stride, f.W],
                                    "values": "normal(0,1)/sqrt(K)"}
    cfg["l2"] = (f"inputs larger than L2 ({touched / 1e9:.2f} GB of algorithmic traffic per step)"
                 if touched > 2 * 126e6 else
                 f"small case: {touched / 1e6:.0f} MB per step, partly L2-resident")
    cfg["peaks"] = {"hbm_gbs": peaks["hbm_gbs"],
                    "f16_tflops": peaks["bf16_tflops"] * F16_PER_BF16, "source": peak_src,
                    "note": "f16 dense peak = measured bf16 burst peak x nominal 1:1 ratio"}
    cfg["seed"] = 0
    return cfg


# --------------------------------------------------------------------------- #
# the GPU arm                                                                 #
# --------------------------------------------------------------------------- #

def setup_device(dev, g: GatherCfg | None, f: FusedCfg | None, device_inputs: bool, seed=0):
    """One symmetric heap holding every member's inputs and outputs; returns
    (heap, offsets, B on the device, host copies of the inputs or None)."""
    import torch

    import gemm_gather_gb300 as gg
    import gg_inputs
    align = 1 << 16
    sizes = []
    if g:
        in_rows = g.W * g.M if g.kind == "all_to_all" else g.M
        sizes += [("g_in", in_rows * g.N * g.es), ("g_out", g.W * g.M * g.N * g.es)]
    if f:
        sizes += [("f_a", f.M * f.K * 2), ("f_out", f.W * f.M * f.N * 2)]
    offs, o = {}, 0
    for name, size in sizes:
        offs[name] = o
        o += (size + align - 1) // align * align
    H = max((c.members()[-1] + 1) for c in (g, f) if c is not None)
    sh = gg.SymmetricHeap(H, o, device=dev)
    gen = gg_inputs.generator(seed, device=dev if device_inputs else "cpu")
    host = None if device_inputs else {"g_in": {}, "f_a": {}}
    if g:
        dt = gg_inputs.DTYPES[g.dtype]
        draw = gg_inputs.uniform_pm1 if g.values == "uniform" else gg_inputs.normal
        in_rows = g.W * g.M if g.kind == "all_to_all" else g.M
        for h in g.members():
            x = draw((in_rows, g.N), dt, gen)
            if host is not None:
                host["g_in"][h] = x
            sh.view(h, offs["g_in"], in_rows, g.N, g.N, dt).copy_(x)
    Bd = None
    if f:
        dt = gg_inputs.DTYPES[f.dtype]
        for h in f.members():
            a = gg_inputs.normal((f.M, f.K), dt, gen, scale=f.K ** -0.5)
            if host is not None:
                host["f_a"][h] = a
            sh.view(h, offs["f_a"], f.M, f.K, f.K, dt).copy_(a)
        B = gg_inputs.normal((f.K, f.N), dt, gen, scale=f.K ** -0.5)
        if host is not None:
            host["B"] = B
        Bd = B.to(dev)
    torch.cuda.synchronize(dev)
    return sh, offs, Bd, host


def max_over_ranks(value: float, device=None) -> float:
    """The slowest rank's value (replicas: the job is as slow as its slowest
    GPU).  A no-op without an initialised process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(roof_step_s: float, ms_per_step: float, world: int) -> float:
    """Percent of one GPU's step roofline, summed over `world` replicas that
    each ran the whole step in the (max-over-ranks) measured time."""
    return 100.0 * world * roof_step_s / (ms_per_step * 1e-3)


def sweep_points(name: str):
    """(GatherCfg | None, FusedCfg | None) points of the configuration sweeps."""
    pts = []
    if name == "budget":  # 8 ranks, 4096x4096 f16, tile 8x256, budget swept, every data path
        for path in ("tma", "bulk", "vector"):
            for p in (8, 16, 32, 64, 148):
                pts.append((replace(GATHER, programs=p, path=path), None))
    elif name == "gather":  # 4 and 8 ranks, M x N x dtype x tile x budget, normal values
        for W in (4, 8):
            for M in (1024, 4096, 16384):
                for N in (4096, 8192):
                    for dt in ("f16", "bf16", "f32"):
                        for bm, bn in ((8, 256), (16, 128), (32, 128)):
                            for p in (64, 128, 148):
                                pts.append((GatherCfg(W=W, M=M, N=N, dtype=dt, bm=bm, bn=bn,
                                                      programs=p, values="normal"), None))
        for M in (1024, 4096, 16384):  # strided subgroup: heaps 1, 3, 5, 7
            for N in (4096, 8192):
                pts.append((GatherCfg(W=4, M=M, N=N, dtype="f16", start=1, stride=2,
                                      values="normal"), None))
    elif name == "small":  # the 2-rank 64x256 f16 case, tile 8x256, 4 programs: launch-bound
        for path in ("tma", "bulk", "vector"):
            pts.append((GatherCfg(W=2, M=64, N=256, programs=4, path=path), None))
    elif name == "variants":  # partitioned all-gather, destination grouping, all-to-all
        for p in (8, 16, 32, 64, 148):
            pts.append((replace(GATHER, programs=p, kind="partitioned", path="tma"), None))
        for path in ("tma", "bulk"):
            for p in (64, 148):
                for gsz in (1, 2, 4):
                    pts.append((replace(GATHER, programs=p, dests_per_wait=gsz, path=path), None))
        for p in (16, 64, 128, 148):
            pts.append((replace(GATHER, programs=p, kind="all_to_all", path="auto"), None))
        for p in (8, 16, 32, 64, 148):  # W single-rank launches in turn
            pts.append((replace(GATHER, programs=p, kind="ranks"), None))
    elif name == "cublas":  # the fused kernel and cuBLAS on the plain GEMM of the same size
        for bn, path in ((512, "auto"), (256, "2sm")):
            for M in (1024, 4096, 16384):
                for dt in ("f16", "bf16"):
                    pts.append((None, replace(FUSED, M=M, dtype=dt, path=path, bn=bn)))
    elif name == "fused":  # 8 ranks, M_local 1024/4096/16384, f16 and bf16, + subgroup (0,2,4)
        for bn, path in ((512, "auto"), (256, "2sm"), (256, "1sm")):
            for M in (1024, 4096, 16384):
                for dt in ("f16", "bf16"):
                    pts.append((None, replace(FUSED, M=M, dtype=dt, path=path, bn=bn)))
            for M in (4096, 16384):
                for dt in ("f16", "bf16"):
                    pts.append((None, replace(FUSED, M=M, dtype=dt, W=4, start=0, stride=2,
                                              path=path, bn=bn)))
    else:
        raise SystemExit(f"unknown sweep {name}")
    return pts


def launch_gather(gg, g: GatherCfg, sh, offs, status, dt, stream):
    """One launch of the configured gather-family collective."""
    args = (sh.heap, -1, sh.ptr(g.start, offs["g_in"]), g.N, sh.ptr(g.start, offs["g_out"]), g.N,
            g.M, g.N, dt, (g.bm, g.bn), g.programs, (g.start, g.stride, g.W))
    if g.kind == "ranks":
        # the pages' single-GPU validation: one launch per logical rank, in turn,
        # each with the whole program budget
        for h in g.members():
            gg.all_gather(sh.heap, h, sh.ptr(h, offs["g_in"]), g.N, sh.ptr(h, offs["g_out"]), g.N,
                          g.M, g.N, dt, (g.bm, g.bn), g.programs, (g.start, g.stride, g.W),
                          status=status, stream=stream, path=g.path)
    elif g.kind == "all_to_all":
        gg.all_to_all(*args, status=status, stream=stream, path=g.path)
    elif g.kind == "partitioned":
        gg.all_gather_partitioned(*args, status=status, stream=stream, path=g.path)
    elif g.dests_per_wait:
        gg.all_gather_grouped(*args, g.dests_per_wait, status=status, stream=stream, path=g.path)
    else:
        gg.all_gather(*args, status=status, stream=stream, path=g.path)


FUSED_REL_TOL = 5e-3  # max |gpu - ref| <= 5e-3 * RMS(ref row) (+ half an ulp of the output type)


def check_point(g: GatherCfg | None, f: FusedCfg | None, sh, offs, Bd) -> str:
    """Check the outputs a sweep point left in the heap; raise on a mismatch.

    Gather family: every member's row block i is, bit for bit, member i's input
    (all-to-all: member i's block d, for member d).  Fused: the W copies of the
    output are bit-identical, and three rows of every rank (first, middle,
    last) are within 5e-3 * RMS(row) plus half an output ulp of a float64
    product computed on the host with torch."""
    import torch

    import gg_inputs
    if g is not None:
        dt = gg_inputs.DTYPES[g.dtype]
        bits = {2: torch.int16, 4: torch.int32}[g.es]
        W, M, N = g.W, g.M, g.N
        in_rows = W * M if g.kind == "all_to_all" else M
        ins = {h: sh.view(h, offs["g_in"], in_rows, N, N, dt).view(bits) for h in g.members()}
        for d_idx, d in enumerate(g.members()):
            out = sh.view(d, offs["g_out"], W * M, N, N, dt).view(bits)
            for i, h in enumerate(g.members()):
                want = ins[h][d_idx * M:(d_idx + 1) * M] if g.kind == "all_to_all" else ins[h]
                if not torch.equal(out[i * M:(i + 1) * M], want):
                    raise RuntimeError(f"{g.describe()}: member {d} block {i} differs")
        return "every block bit-exact"
    dt = gg_inputs.DTYPES[f.dtype]
    W, M, N, K = f.W, f.M, f.N, f.K
    first = sh.view(f.members()[0], offs["f_out"], W * M, N, N, dt)
    for d in f.members()[1:]:
        if not torch.equal(sh.view(d, offs["f_out"], W * M, N, N, dt).view(torch.int16),
                           first.view(torch.int16)):
            raise RuntimeError(f"{f.describe()}: member {d}'s copy differs from member "
                               f"{f.members()[0]}'s")
    rows = sorted({0, M // 2, M - 1})
    b64 = Bd.to("cpu", torch.float64)
    mant = 10 if f.dtype == "f16" else 7
    for i, h in enumerate(f.members()):
        a = sh.view(h, offs["f_a"], M, K, K, dt)[rows].to("cpu", torch.float64)
        ref = a @ b64
        got = first[[i * M + r for r in rows]].to("cpu", torch.float64)
        rms = ref.pow(2).mean(dim=1, keepdim=True).sqrt()
        mag = torch.maximum(ref.abs(), got.abs()).clamp_min(2.0 ** -14)
        half_ulp = torch.exp2(torch.floor(torch.log2(mag)) - mant - 1)
        bad = (got - ref).abs() > FUSED_REL_TOL * rms + half_ulp
        if bool(bad.any()):
            raise RuntimeError(f"{f.describe()}: rank {h}: {int(bad.sum())} values outside "
                               "the tolerance")
    return "copies bit-identical; 3 rows per rank within tolerance of a float64 product"


def run_sweep(args):
    """Time each point of a sweep in this process; one JSON line per point."""
    import torch

    import gemm_gather_gb300 as gg
    import gg_inputs
    if args.claims is not None:
        gg.set_claim_policy(args.claims)
    if args.store_policy is not None:
        gg.set_store_policy(args.store_policy)
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for g, f in sweep_points(args.sweep):
        if args.only and not any(o in (g or f).describe() for o in args.only.split("|")):
            continue
        # --gather / --fused overrides apply to every point of the sweep
        g = parse_cfg(args.gather, g) if g else None
        f = parse_cfg(args.fused, f) if f else None
        if f and f.programs == 0:
            f.programs = sms
        sh, offs, Bd, _ = setup_device(dev, g, f, device_inputs=True)
        status = torch.zeros(1, dtype=torch.int32, device=dev)

        def launch():
            if g:
                launch_gather(gg, g, sh, offs, status, gg_inputs.DTYPES[g.dtype], None)
            else:
                gg.matmul_all_gather(sh.heap, -1, sh.ptr(f.start, offs["f_a"]), f.K, Bd, f.N,
                                     sh.ptr(f.start, offs["f_out"]), f.N, f.M, f.N, f.K,
                                     gg_inputs.DTYPES[f.dtype], f.tile, f.programs,
                                     (f.start, f.stride, f.W), status=status, path=f.path)

        t_rg, t_rf = roofline_times(peaks, g, f)
        work = t_rg + t_rf

        def timed(fn):
            """(median ms per launch over the repeats, launches per run, clocks)"""
            steps = int(max(5, min(args.steps, 0.5 / max(work, 1e-6))))
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize(dev)
            clocks = ClockSampler(dev.index or 0, None) if args.sweep_clocks else None
            if clocks:
                clocks.start()
                steps = max(steps, int(1.0 / max(work, 1e-6)))  # at least ~1 s under load
            runs = []
            for _ in range(max(1, args.repeats)):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(steps):
                    fn()
                e1.record()
                torch.cuda.synchronize(dev)
                runs.append(e0.elapsed_time(e1) / steps)
            return runs, steps, (clocks.stop() if clocks else None)

        gg.set_trace(True)  # the kernel's own SM clock, from its last timed launch
        runs, steps, clk = timed(launch)
        trace = gg.trace_read()
        gg.set_trace(False)
        ms = statistics.median(runs)
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())}")
        checked = check_point(g, f, sh, offs, Bd)
        rec = {"sweep": args.sweep, "workload": (g or f).describe(), "ms": ms, "steps": steps,
               "runs_ms": runs, "roofline_ms": 1e3 * work, "frac": 1e3 * work / ms,
               "checked": checked}
        moved = gather_bytes(g) if g else fused_bytes(f)
        if moved < 2 * L2_BYTES and args.sweep != "small":
            # small enough to be partly L2-resident between back-to-back launches:
            # time it again with a buffer larger than L2 written before every launch
            flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
            tot = 0.0
            n_fl = max(5, min(steps, 50))
            for _ in range(n_fl):
                flush.fill_(1)
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record()
                launch()
                a1.record()
                a1.synchronize()
                tot += a0.elapsed_time(a1)
            rec["ms_l2_flushed"] = tot / n_fl
            rec["frac_l2_flushed"] = 1e3 * work / rec["ms_l2_flushed"]
            del flush
        if args.sweep == "small":
            # the same launches replayed from a CUDA graph (no per-launch host work)
            cap = torch.cuda.Stream(dev)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                for _ in range(100):
                    launch()
            graph.replay()
            torch.cuda.synchronize(dev)
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record()
            for _ in range(10):
                graph.replay()
            g1.record()
            torch.cuda.synchronize(dev)
            rec["us_per_launch"] = 1e3 * ms
            rec["graph_us_per_launch"] = g0.elapsed_time(g1) / 1000 * 1e3
        kclk = kernel_clock(trace["all_gather" if g else "matmul_all_gather"])
        if kclk:
            if f:
                sms = torch.cuda.get_device_properties(dev).multi_processor_count
                kclk["per_clock_frac"] = fused_flops(f) / (kclk["cycles"] * sms *
                                                           TC_FLOP_PER_SM_CYCLE)
            rec["kernel_clock"] = kclk
        if clk:
            rec["clocks"] = clk
            if f:
                tcs = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * F16_PER_BF16
                rec["frac_of_sustained_peak"] = fused_flops(f) / (ms * 1e-3) / 1e12 / tcs
        if g:
            rec["GB/s"] = gather_bytes(g) / (ms * 1e-3) / 1e9
        else:
            rec["TFLOP/s"] = fused_flops(f) / (ms * 1e-3) / 1e12
        if args.sweep == "cublas":
            # cuBLAS (torch.matmul) on the plain GEMM of the same total size, one
            # output copy, timed the same way right after, on the same GPU
            dt = gg_inputs.DTYPES[f.dtype]
            a_all = torch.randn(f.W * f.M, f.K, device=dev, dtype=torch.float32).mul_(
                f.K ** -0.5).to(dt)
            c_all = torch.empty(f.W * f.M, f.N, device=dev, dtype=dt)
            c_runs, _, c_clk = timed(lambda: torch.matmul(a_all, Bd, out=c_all))
            c_ms = statistics.median(c_runs)
            rec["cublas"] = {"gemm": f"{f.W * f.M}x{f.N}x{f.K} {f.dtype}", "ms": c_ms,
                             "TFLOP/s": fused_flops(f) / (c_ms * 1e-3) / 1e12, "clocks": c_clk}
            rec["vs_cublas"] = c_ms / ms
            del a_all, c_all
        print(json.dumps(rec), flush=True)
        del sh, Bd, status
        torch.cuda.empty_cache()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--workload", default="step", choices=["step", "gather", "fused"],
                    help="step: the all-gather then the fused kernel; or one of them alone")
    ap.add_argument("--preset", default="largest", choices=sorted(PRESETS),
                    help="largest: W=8 16384x8192 f32 all-gather + fused M_local=16384 "
                    "(default); small: W=8 4096x4096 f16 all-gather + fused M_local=1024")
    ap.add_argument("--gather", default="", help="overrides, e.g. W=4,M=1024,N=8192,dtype=f32,"
                    "tile=16x128,programs=128,group=1:2,values=normal,path=bulk")
    ap.add_argument("--fused", default="", help="overrides, e.g. M=16384,dtype=bf16,group=0:2,W=4")
    ap.add_argument("--e2e-steps", type=int, default=20, help="0 skips the end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--device-inputs", default="auto", choices=["auto", "yes", "no"],
                    help="draw inputs on the GPU (seeded) instead of the CPU")
    ap.add_argument("--clocks-out", default=None)
    ap.add_argument("--sweep", default=None,
                    choices=["budget", "gather", "fused", "variants", "small", "cublas"],
                    help="time every point of a configuration sweep (one JSON line each)")
    ap.add_argument("--only", default="", help="sweep: run only points whose description "
                    "contains one of these '|'-separated substrings")
    ap.add_argument("--repeats", type=int, default=3,
                    help="sweep: timed runs per point; the median is reported")
    ap.add_argument("--sweep-clocks", action="store_true",
                    help="sample SM clocks while each sweep point runs (about 1 s per point)")
    ap.add_argument("--store-policy", default=None, choices=["plain", "evict_first"],
                    help="L2 hint on the gather family's stores (default: the library's, "
                    "evict_first)")
    ap.add_argument("--claims", default=None, choices=["auto", "always", "never"],
                    help="which gather launches claim runs of tiles from the heap's workspace "
                    "(default: the library's, auto)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "mine" and os.environ.get("GEMM_GATHER_CHECKED", "0") == "1":
        # the checked build bounds every access of the gather kernels: a
        # development build whose times would not describe the library
        ap.error("GEMM_GATHER_CHECKED=1 loads the checked build, which is not for measurement")
    if args.sweep:
        return run_sweep(args)
    base_g, base_f = PRESETS[args.preset]
    g = parse_cfg(args.gather, base_g) if args.workload in ("step", "gather") else None
    f = parse_cfg(args.fused, base_f) if args.workload in ("step", "fused") else None
    peaks, peak_src = load_peaks()
    if args.impl == "reference":
        return run_reference(args, peaks, peak_src, g, f)

    import torch
    import torch.distributed as dist

    import gemm_gather_gb300 as gg
    import gg_inputs

    if args.claims is not None:
        gg.set_claim_policy(args.claims)
    if args.store_policy is not None:
        gg.set_store_policy(args.store_policy)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if f and f.programs == 0:
        f.programs = sms
    in_bytes = (g.W * g.M * g.N * g.es if g else 0) + (f.W * f.M * f.K * 2 if f else 0)
    device_inputs = args.device_inputs == "yes" or (args.device_inputs == "auto"
                                                   and in_bytes > (1 << 30))
    sh, offs, Bd, host = setup_device(dev, g, f, device_inputs)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    gdt = gg_inputs.DTYPES[g.dtype] if g else None
    g_in_rows = (g.W * g.M if g.kind == "all_to_all" else g.M) if g else 0
    fdt = gg_inputs.DTYPES[f.dtype] if f else None

    def launch_step(heap, b_dev, strm):
        """The two kernels of one step on `heap` (a SymmetricHeap) and stream `strm`."""
        if g:
            launch_gather(gg, g, heap, offs, status, gdt, strm)
        if f:
            gg.matmul_all_gather(heap.heap, -1, heap.ptr(f.start, offs["f_a"]), f.K, b_dev, f.N,
                                 heap.ptr(f.start, offs["f_out"]), f.N, f.M, f.N, f.K, fdt,
                                 f.tile, f.programs, (f.start, f.stride, f.W),
                                 status=status, stream=strm, path=f.path)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if g:
            launch_gather(gg, g, sh, offs, status, gdt, stream)
        if ev is not None:
            ev[1].record(stream)
        if f:
            gg.matmul_all_gather(sh.heap, -1, sh.ptr(f.start, offs["f_a"]), f.K, Bd, f.N,
                                 sh.ptr(f.start, offs["f_out"]), f.N, f.M, f.N, f.K, fdt,
                                 f.tile, f.programs, (f.start, f.stride, f.W),
                                 status=status, stream=stream, path=f.path)
        if ev is not None:
            ev[2].record(stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # each kernel's first CTA records its start/end wall time and SM cycles (four
    # 8-byte stores per launch): the clock the kernel itself ran at
    gg.set_trace(True)
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
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    barrier()
    clk = clocks.stop() if clocks else None
    trace = gg.trace_read(stream)  # the last timed launch of each kernel
    gg.set_trace(False)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the timed steps")
    elapsed_ms = t_start.elapsed_time(t_end)
    g_all = [e[0].elapsed_time(e[1]) for e in evs] if g else [0.0]
    f_all = [e[1].elapsed_time(e[2]) for e in evs] if f else [0.0]
    g_ms, f_ms = statistics.mean(g_all), statistics.mean(f_all)

    def spread(xs):  # per-launch statistics of one kernel over the timed steps
        return {"median": statistics.median(xs), "min": min(xs), "max": max(xs)}
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    ms_step = elapsed_ms / args.steps

    # ---- end to end through the C ABI, host buffers, copies in the timed region
    e2e = None
    if args.e2e_steps > 0:
        try:
            if host is None:
                # inputs were drawn on the device: stage them once into pinned host memory
                def pinned_copy(t):
                    p = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    p.copy_(t)
                    return p

                pin = {"g_in": {}, "f_a": {}}
                if g:
                    for h in g.members():
                        pin["g_in"][h] = pinned_copy(sh.view(h, offs["g_in"], g_in_rows, g.N, g.N,
                                                             gdt))
                if f:
                    for h in f.members():
                        pin["f_a"][h] = pinned_copy(sh.view(h, offs["f_a"], f.M, f.K, f.K, fdt))
                pin_b = pinned_copy(Bd) if f else None
            else:
                pin = {k: {h: x.pin_memory() for h, x in v.items()} for k, v in host.items()
                       if k != "B"}
                pin_b = host["B"].pin_memory() if f else None
            host = None

            # The step's result: the gathered outputs.  Every member holds an identical
            # copy (what the parity tests check), so the result is read from the first
            # member; the variant that reads all W copies is timed as well.
            def out_set(members_g, members_f):
                og = {h: torch.empty((g.W * g.M, g.N), dtype=gdt).pin_memory()
                      for h in members_g}
                of = {h: torch.empty((f.W * f.M, f.N), dtype=fdt).pin_memory()
                      for h in members_f}
                return og, of

            first_g = g.members()[:1] if g else []
            first_f = f.members()[:1] if f else []
            outs = [out_set(first_g, first_f), out_set(first_g, first_f)]
            h2d = sum(x.numel() * x.element_size() for v in pin.values() for x in v.values()) + \
                (pin_b.numel() * 2 if f else 0)

            def nbytes(oset):
                return sum(x.numel() * x.element_size() for d in oset for x in d.values())

            d2h = nbytes(outs[0])
            # every member's copy as well, while it fits a bounded pinned buffer
            d2h_all = (g.W * g.W * g.M * g.N * g.es if g else 0) + \
                (f.W * f.W * f.M * f.N * 2 if f else 0)
            outs_all = ([out_set(g.members() if g else [], f.members() if f else [])] * 2
                        if d2h_all <= E2E_ALL_COPIES_MAX_BYTES else None)

            def copy_in(heap, b_dev):
                if g:
                    for h in g.members():
                        heap.view(h, offs["g_in"], g_in_rows, g.N, g.N, gdt).copy_(pin["g_in"][h],
                                                                                    non_blocking=True)
                if f:
                    for h in f.members():
                        heap.view(h, offs["f_a"], f.M, f.K, f.K, fdt).copy_(pin["f_a"][h],
                                                                             non_blocking=True)
                    b_dev.copy_(pin_b, non_blocking=True)

            def copy_out(heap, oset):
                og, of = oset
                for h, o in og.items():
                    o.copy_(heap.view(h, offs["g_out"], g.W * g.M, g.N, g.N, gdt), non_blocking=True)
                for h, o in of.items():
                    o.copy_(heap.view(h, offs["f_out"], f.W * f.M, f.N, f.N, fdt), non_blocking=True)

            e2e_steps = max(1, min(args.e2e_steps, args.steps))

            # (1) serial: copy in, compute, copy out, one step after the other, one stream
            def serial_step():
                copy_in(sh, Bd)
                launch_step(sh, Bd, stream)
                copy_out(sh, outs[0])

            for _ in range(3):
                serial_step()
            barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(e2e_steps):
                serial_step()
            e1.record(stream)
            barrier()
            serial_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)

            # (2) pipelined: two device buffer sets; step i copies in on one stream,
            # computes on another and copies out on a third, overlapping steps i-1
            # and i+1 (every step still moves all of its inputs and outputs)
            sh2 = gg.SymmetricHeap(sh.H, sh.part_bytes, device=dev)
            bufs = [(sh, Bd), (sh2, torch.empty_like(Bd) if f else None)]
            s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
            ev_in = [torch.cuda.Event() for _ in range(2)]
            ev_cmp = [torch.cuda.Event() for _ in range(2)]
            ev_out = [torch.cuda.Event() for _ in range(2)]

            run_kernels = [True]

            def pipelined(n, out_sets):
                for i in range(n):
                    b = i % 2
                    heap, b_dev = bufs[b]
                    with torch.cuda.stream(s_in):
                        if i >= 2:
                            s_in.wait_event(ev_cmp[b])  # step i-2 no longer reads these inputs
                        copy_in(heap, b_dev)
                        ev_in[b].record(s_in)
                    with torch.cuda.stream(s_cmp):
                        s_cmp.wait_event(ev_in[b])
                        if i >= 2:
                            s_cmp.wait_event(ev_out[b])  # step i-2's outputs are copied out
                        if run_kernels[0]:
                            launch_step(heap, b_dev, s_cmp)
                        ev_cmp[b].record(s_cmp)
                    with torch.cuda.stream(s_out):
                        s_out.wait_event(ev_cmp[b])
                        copy_out(heap, out_sets[b])
                        ev_out[b].record(s_out)

            def timed_pipeline(out_sets):
                pipelined(3, out_sets)
                barrier()
                p0 = torch.cuda.Event(enable_timing=True)
                p1 = torch.cuda.Event(enable_timing=True)
                p0.record(s_in)
                pipelined(e2e_steps, out_sets)
                p1.record(s_out)
                barrier()
                return max_over_ranks(p0.elapsed_time(p1) / e2e_steps, dev)

            e2e_ms = timed_pipeline(outs)
            # the same pipelined copies with no kernels: the host link's share of the step
            run_kernels[0] = False
            copies_ms = timed_pipeline(outs)
            run_kernels[0] = True
            if outs_all is not None:
                all_copies = {"d2h_bytes_per_step": d2h_all, "ms_per_step": timed_pipeline(outs_all)}
            else:
                all_copies = {"d2h_bytes_per_step": d2h_all, "ms_per_step": None,
                              "skipped": f"more than {E2E_ALL_COPIES_MAX_BYTES >> 30} GiB of pinned "
                                         "host memory"}
            e2e = {"h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                   "steps": e2e_steps, "serial_ms_per_step": serial_ms,
                   "copies_only": {"ms_per_step": copies_ms,
                                   "GB/s": (h2d + d2h) / (copies_ms * 1e-3) / 1e9,
                                   "note": "the same pipelined host<->device copies with no kernels"},
                   "all_copies": all_copies,
                   "path": ("pinned host -> heap (cudaMemcpyAsync) -> C-ABI calls -> pinned host; "
                            "every member's inputs copied in, the gathered outputs read back from "
                            "member 0 (all members hold identical copies); steps pipelined over two "
                            "device buffer sets and three streams; all_copies reads every member's "
                            "output")}
            del sh2, bufs
        except (RuntimeError, MemoryError) as exc:
            # a failed end-to-end leg (e.g. pinned host memory exhausted) must not
            # cost the device-timed line: report it instead (one process only;
            # with replicas the other ranks would wait at the leg's barriers)
            if world > 1:
                raise
            torch.cuda.synchronize(dev)
            e2e = {"ms_per_step": None, "error": f"{type(exc).__name__}: {exc}"[:300]}

    # ---- roofline bookkeeping
    t_rg, t_rf = roofline_times(peaks, g, f)
    roof_step = t_rg + t_rf
    value = whole_job_value(roof_step, ms_step, world)
    if e2e and e2e.get("ms_per_step"):
        e2e = {"value": whole_job_value(roof_step, e2e["ms_per_step"], world), "unit": UNIT, **e2e}
    elif e2e:
        e2e = {"value": None, "unit": UNIT, **e2e}
    hbm_peak = peaks["hbm_gbs"]
    tc_peak = peaks["bf16_tflops"] * F16_PER_BF16
    kernels = {}
    if g:
        g_gbs = gather_bytes(g) / (g_ms * 1e-3) / 1e9
        kname = {"vector": "ag_vec_kernel", "bulk": "ag_bulk_kernel"}.get(g.path, "ag_tma_kernel")
        kernels["all_gather"] = {"kernel": kname, "ms": g_ms, "ms_per_launch": spread(g_all),
                                 "clock": kernel_clock(trace["all_gather"]),
                                 "GB/s": g_gbs,
                                 "roofline_ms": 1e3 * t_rg, "frac": g_gbs / hbm_peak,
                                 "bound": "hbm", "algorithmic_bytes": gather_bytes(g),
                                 "traffic": traffic_for(kname, "ag_kernels.cu", g.describe())}
    if f:
        f_tfs = fused_flops(f) / (f_ms * 1e-3) / 1e12
        chosen = gg.matmul_all_gather_plan(sh.heap, -1, sh.ptr(f.start, offs["f_a"]), f.K, Bd, f.N,
                                           sh.ptr(f.start, offs["f_out"]), f.N, f.M, f.N, f.K,
                                           fdt, f.tile, f.programs,
                                           (f.start, f.stride, f.W), f.path)
        fk = "mag1_kernel" if chosen == "1sm" else ("mag2w_kernel" if f.bn == 512 else
                                                     "mag2_kernel")
        fclk = kernel_clock(trace["matmul_all_gather"])
        if fclk:
            # work per SM cycle against the tensor pipes' nominal dense rate
            fclk["per_clock_frac"] = fused_flops(f) / (fclk["cycles"] * sms * TC_FLOP_PER_SM_CYCLE)
            fclk["per_clock_note"] = (f"FLOPs / (SM cycles of the traced launch x {sms} SMs x "
                                      f"{TC_FLOP_PER_SM_CYCLE} dense f16 FLOP per SM cycle)")
        kernels["matmul_all_gather"] = {"kernel": fk, "ms": f_ms, "ms_per_launch": spread(f_all),
                                        "clock": fclk,
                                        "TFLOP/s": f_tfs,
                                        "roofline_ms": 1e3 * t_rf, "frac": f_tfs / tc_peak,
                                        "bound": "tensor", "algorithmic_flops": fused_flops(f),
                                        "algorithmic_bytes": fused_bytes(f),
                                        "traffic": traffic_for(fk, "mag_kernel.cu", f.describe()),
                                        "programs": f.programs}
    if g and (not f or g_ms >= f_ms):
        k = kernels["all_gather"]
        roof = {"kernel": k["kernel"], "bound": "hbm", "achieved": k["GB/s"], "peak": hbm_peak,
                "unit": "GB/s", "frac": k["frac"],
                "traffic": traffic_for(k["kernel"], "ag_kernels.cu", g.describe()),
                "per_unit": "bytes = W*M*N*s reads + W^2*M*N*s writes per launch"}
    else:
        k = kernels["matmul_all_gather"]
        roof = {"kernel": k["kernel"], "bound": "tensor", "achieved": k["TFLOP/s"],
                "peak": tc_peak, "unit": "TFLOP/s", "frac": k["frac"],
                "traffic": traffic_for(k["kernel"], "mag_kernel.cu", f.describe()),
                "per_unit": "FLOPs = 2*W*M*N*K per launch"}
    roof["peak_source"] = ("measured (MEASURED_PEAKS.json)" if peak_src == "measured"
                           else "fallback")
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    cpu = None if args.no_cpu_baseline else cpu_baseline(peaks, g, f)
    dtypes = sorted({c.dtype for c in (g, f) if c is not None})
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "+".join(dtypes), "data": "synthetic",
        "config": config_block(peaks, peak_src, g, f),
        "kernels": kernels,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": (int(g is not None) + int(f is not None)) * args.steps,
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
