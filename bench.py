#!/usr/bin/env python3
"""Benchmark of the conv2d input gradient (implicit GEMM) on GB300.

Metric: dgrad TFLOP/s (useful FLOPs 2*N*Co*OH*OW*Ci*kH*kW) and the fraction of
the kernel's roofline, on the ResNet 3x3 workload (N=32, Ci=Co=64, 56x56,
stride 1, pad 1, bf16 in, float32 out) unless --config names another.

One step = one pass of the whole path over one batch: the weight pre-pack
kernel, then the dgrad kernel (or the dgrad kernel alone where it packs the
weights in shared memory itself: the workspace size is then 0).  Inputs are resident in HBM; every step uses
the next of several buffer sets whose total exceeds 3x the L2 cache, so each
step starts cold.  The timed region replays a CUDA graph of exactly K such
steps (no event nodes inside the graph, so each kernel's prologue can overlap
the previous kernel's tail), then a graph of back-to-back dgrad launches alone
for the kernel's per-launch time; it is bracketed by a barrier and
synchronisation on both sides.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle (the
only reference there is) on a bounded sample of the same workload instead.
Multi-GPU (torchrun): data parallel over the batch.  The global batch is
N x world images; rank r takes its own shard of N of them (shard_bounds), a
replica of the weights, and writes its own slice of grad_in -- no collective on
the data path (weak scaling: per-rank work is fixed).  value = all ranks' FLOPs
/ the slowest rank's time.

``--profile-launches L`` only launches the dgrad kernel L times over the
rotating buffer sets (for an ncu capture of per-launch DRAM traffic), and
``--record-traffic CSV`` turns that capture's CSV into the workload's traffic
record under profiles/.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dgrad TFLOP/s and % of dense tensor-core roofline per config (1 GB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ("conv2d_backward_implicit_gb300/csrc/dgrad_tc.cu",
                  "conv2d_backward_implicit_gb300/csrc/dgrad_internal.h",
                  "conv2d_backward_implicit_gb300/csrc/plan.cu")


# ------------------------------------------------------------------ helpers
def useful_flops(wl) -> float:
    return 2.0 * wl.N * wl.Co * wl.OH * wl.OW * wl.Ci * wl.kH * wl.kW


def algorithmic_bytes(wl) -> int:
    """grad_out + weight + grad_in, each moved once (no materialised im2col)."""
    esize = 4 if wl.dtype == "f32" else 2
    go = wl.N * wl.Co * wl.OH * wl.OW * esize
    w = wl.Co * wl.Ci * wl.kH * wl.kW * esize
    gi = wl.N * wl.Ci * wl.H * wl.W * 4
    return go + w + gi


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def code_of(source: str) -> str:
    """The source without comments and blank lines: edits to comments alone
    leave the compiled kernel, and so its fingerprint, unchanged."""
    source = re.sub(r"/\*.*?\*/", "", source, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in source.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_fingerprint() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(config_key: str):
    """dram bytes per launch from a committed ncu summary, if it is for this kernel source."""
    path = os.path.join(ROOT, "profiles", f"dgrad_tc_{config_key}.traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_fingerprint") != kernel_fingerprint():
        return None
    return d.get("dram_bytes_per_launch")


def shard_bounds(global_n: int, world: int, rank: int):
    """[lo, hi) of the global batch that `rank` processes: contiguous shards,
    sizes differing by at most one, together covering [0, global_n) once."""
    base, extra = divmod(global_n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def measure_tf32_peak(dev, n: int = 8192, reps: int = 10) -> float:
    """Dense TF32 tensor-core rate (TFLOP/s): torch.matmul of float32 n x n
    matrices with TF32 allowed, best of `reps` after a warm-up (the method of
    the measured bf16 peak, for the dtype the fp32 workloads compute in)."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(n, n, device=dev)
        b = torch.randn(n, n, device=dev)
        c = torch.empty(n, n, device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        torch.cuda.synchronize(dev)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b, c
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


_UNIT = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "nsecond": 1e-9, "ns": 1e-9,
         "usecond": 1e-6, "us": 1e-6, "msecond": 1e-3, "ms": 1e-3, "second": 1.0, "s": 1.0}


def traffic_from_ncu_csv(text: str, kernel_pattern: str = "dgrad_tc_kernel"):
    """Per-launch DRAM bytes of the kernel from an ncu --csv log of the metrics
    dram__bytes_read.sum, dram__bytes_write.sum and gpu__time_duration.sum:
    [(launch id, kernel name, read bytes, write bytes, seconds)], in launch order."""
    import csv
    import io
    lines = [ln for ln in text.splitlines() if ln.startswith('"')]
    rows = list(csv.DictReader(io.StringIO("\n".join(lines))))
    per = {}
    for r in rows:
        name = r.get("Kernel Name", "")
        if kernel_pattern not in name:
            continue
        metric, unit = r.get("Metric Name", ""), r.get("Metric Unit", "").strip().lower()
        try:
            value = float(r.get("Metric Value", "").replace(",", ""))
        except ValueError:
            continue
        value *= _UNIT.get(unit, 1.0)
        key = int(r["ID"])
        d = per.setdefault(key, {"name": name})
        if metric == "dram__bytes_read.sum":
            d["read"] = value
        elif metric == "dram__bytes_write.sum":
            d["write"] = value
        elif metric == "gpu__time_duration.sum":
            d["seconds"] = value
    out = []
    for key in sorted(per):
        d = per[key]
        if "read" in d and "write" in d:
            out.append((key, d["name"], int(d["read"]), int(d["write"]), d.get("seconds")))
    return out


def traffic_record(launches, wl, key, command: str):
    """The traffic record of a workload: DRAM bytes per launch averaged over
    the captured launches after the first (steady state: a launch's grad_in
    writes leave L2 during later launches, so the first one shows only reads)."""
    steady = launches[1:] if len(launches) > 1 else launches
    rd = round(sum(x[2] for x in steady) / len(steady))
    wr = round(sum(x[3] for x in steady) / len(steady))
    alg = algorithmic_bytes(wl)
    return {
        "kernel": launches[0][1].split("(")[0].replace("void ", "").strip(),
        "workload": workload_config(wl, key, "")["workload"],
        "kernel_fingerprint": kernel_fingerprint(),
        "dram_bytes_per_launch": int(rd + wr),
        "dram_read_bytes": int(rd),
        "dram_write_bytes": int(wr),
        "algorithmic_bytes": alg,
        "traffic_over_algorithmic": (rd + wr) / alg,
        "launches_averaged": len(steady),
        "per_launch": [{"id": x[0], "read": x[2], "write": x[3], "us": (x[4] or 0) * 1e6}
                       for x in launches],
        "note": "steady-state DRAM traffic per launch: ncu with --cache-control none over "
                "back-to-back launches on rotating buffer sets, averaged over the launches "
                "after the first (whose grad_in writes are still in L2 when it ends)",
        "command": command,
    }


def reduce_max(value: float, dist_on: bool, device=None) -> float:
    """Max of a scalar over ranks (identity when not distributed)."""
    if not dist_on:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(flops_per_rank: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank's useful FLOPs over the slowest rank's time."""
    return flops_per_rank * steps * world / (max_ms * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=timestamp," + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        t0, t1 = self.window or (0, float("inf"))
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 1 + len(self.FIELDS):
                continue
            rows.append((ts, parts))
        inside = [r for ts, r in rows if t0 - 0.06 <= ts <= t1 + 0.06]
        use = inside if inside else rows[-5:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in use if num(r[1]) is not None]
        mx = [num(r[2]) for r in use if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------ CPU oracle legs
def oracle_sample(wl, planes_per_step: int, steps: int, warmup: int):
    """Time the oracle on `steps` samples of one image x `planes_per_step` input channels."""
    import numpy as np
    import oracle
    from conv2d_backward_implicit_gb300 import workloads
    one = wl.with_batch(1)
    g, w = workloads.make_inputs(one, seed=0)
    g = g.double().numpy()
    w = w.double().numpy()
    cs = max(1, min(planes_per_step, wl.Ci))
    ws = [np.ascontiguousarray(w[:, (k * cs) % wl.Ci:(k * cs) % wl.Ci + cs])
          for k in range(max(1, wl.Ci // cs))]
    ws = [x for x in ws if x.shape[1] == cs] or [np.ascontiguousarray(w[:, :cs])]
    threads = 0
    for i in range(warmup):
        oracle.dgrad(g, ws[i % len(ws)], wl.H, wl.W, wl.stride, wl.padding_h, wl.padding_w)
    t0 = time.perf_counter()
    for i in range(steps):
        _, threads = oracle.dgrad(g, ws[i % len(ws)], wl.H, wl.W, wl.stride, wl.padding_h,
                                  wl.padding_w, return_threads=True)
    dt = time.perf_counter() - t0
    flops = 2.0 * wl.Co * wl.OH * wl.OW * cs * wl.kH * wl.kW * steps
    return flops, dt, threads, cs


def cpu_baseline(wl, budget_s: float = 12.0):
    """The oracle as it stands on the host cores: whole images, repeated for ~budget_s."""
    flops1, dt1, threads, _ = oracle_sample(wl, wl.Ci, 1, 0)
    reps = max(1, min(int(budget_s / max(dt1, 1e-3)), 2000))
    flops, dt, threads, _ = oracle_sample(wl, wl.Ci, reps, 0)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{reps} x one image (all {wl.Ci} input channels) of the {wl.name} "
                      f"workload, {dt:.1f} s of CPU time"}


def run_reference(args, wl, key):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # Size each step so the whole run stays within about two minutes.
    probe_flops, probe_dt, _, _ = oracle_sample(wl, 16, 1, 0)
    per_plane = probe_dt / 16.0
    total_budget = 90.0
    planes = int(total_budget / max(1, args.steps + args.warmup) / max(per_plane, 1e-6))
    planes = max(1, min(planes, wl.Ci))
    flops, dt, threads, cs = oracle_sample(wl, planes, args.steps, args.warmup)
    value = flops / dt / 1e12
    sample = (f"each step: one image x {cs} of {wl.Ci} input channels of the {wl.name} workload "
              f"(double-precision direct loop)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, same recipe as the GPU arm)",
        "config": workload_config(wl, key, l2_note="CPU oracle"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, key, l2_note):
    return {"workload": f"{wl.name}: N={wl.N} Ci={wl.Ci} Co={wl.Co} H=W={wl.H} "
                        f"k={wl.kH}x{wl.kW} s={wl.stride} p={wl.padding_h},{wl.padding_w} "
                        f"{wl.dtype} in, f32 out",
            "key": key, "N": wl.N, "Ci": wl.Ci, "Co": wl.Co, "H": wl.H, "W": wl.W,
            "kernel": [wl.kH, wl.kW], "stride": wl.stride,
            "padding": [wl.padding_h, wl.padding_w], "out": [wl.OH, wl.OW],
            "input_dtype": wl.dtype, "l2": l2_note}


# ------------------------------------------------------------------ GPU arm
def kernel_only(dg, workloads, wl, key, dev, stream, launches=600):
    """Per-launch time of the dgrad kernel alone on one workload: cold L2 via
    rotating buffer sets (> 3x L2), weights packed beforehand, a CUDA graph of
    back-to-back launches timed with events; returns the roofline figures."""
    import torch
    g_cpu, w_cpu = workloads.make_inputs(wl, seed=0)
    p = dg.params_from_shapes(g_cpu.shape, w_cpu.shape, wl.H, wl.W, wl.stride, wl.padding_h,
                              wl.padding_w)
    code = dg.DTYPE_CODE[wl.dtype]
    kernel = dg.conv2d_grad_input_select_kernel(p, code)
    ws = dg.conv2d_grad_input_workspace_size(p, code)
    alg = algorithmic_bytes(wl)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 * 2**20)
    # (capped: a workload of a few KB, e.g. the tiny one, is launch-latency bound
    # and measured L2-resident)
    n_sets = min(max(2, math.ceil(3 * l2 / alg)), 512)
    sets = []
    for _ in range(n_sets):
        s = {"g": g_cpu.to(dev), "out": torch.empty(wl.grad_in_shape, device=dev, dtype=torch.float32)}
        if ws > 0:
            s["src"] = torch.empty(ws, dtype=torch.uint8, device=dev)
            dg.conv2d_grad_input_pack_weight(w_cpu.to(dev), s["src"], ws, p, code, stream)
        else:  # CUDA-core kernel, or a kernel that packs the weights itself
            s["src"] = w_cpu.to(dev)
        sets.append(s)
    stream.synchronize()

    def launch_all():
        for s in sets:
            dg.conv2d_grad_input_prepacked(s["g"], s["src"], s["out"], p, code, stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            launch_all()
    stream.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        launch_all()
    reps = max(1, launches // n_sets)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        gr.replay()
        e0.record(stream)
        for _ in range(reps):
            gr.replay()
        e1.record(stream)
    stream.synchronize()
    rc = dg.conv2d_grad_input_check_errors(stream)
    if rc != 0:
        raise RuntimeError(f"{key}: {dg.conv2d_grad_input_status_string(rc)}")
    k_ms = e0.elapsed_time(e1) / (reps * n_sets)
    del sets, gr
    return k_ms, alg, kernel


def forward_call(dg, workloads, wl, dev, stream, calls=300):
    """The stride-1 forward convolution of the layer (conv2d_forward: weight
    flip, pack unless the kernel packs itself, kernel; stream-ordered workspace)
    on rotating buffer sets
    (> 3x L2), back to back, timed with events; returns ms per call."""
    import torch
    gen = torch.Generator().manual_seed(0)
    tdt = workloads.TORCH_DTYPE[wl.dtype]
    x_cpu = torch.randn((wl.N, wl.Ci, wl.H, wl.W), generator=gen).to(tdt)
    w_cpu = (torch.randn(wl.weight_shape, generator=gen) * wl.w_std).to(tdt)
    p = dg.params_from_shapes((wl.N, wl.Co, wl.OH, wl.OW), w_cpu.shape, wl.H, wl.W, wl.stride,
                              wl.padding_h, wl.padding_w)
    code = dg.DTYPE_CODE[wl.dtype]
    esize = 4 if wl.dtype == "f32" else 2
    nbytes = x_cpu.numel() * esize + w_cpu.numel() * esize + wl.N * wl.Co * wl.OH * wl.OW * 4
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 * 2**20)
    n_sets = min(max(2, math.ceil(3 * l2 / nbytes)), 512)
    sets = [(x_cpu.to(dev), w_cpu.to(dev),
             torch.empty((wl.N, wl.Co, wl.OH, wl.OW), device=dev, dtype=torch.float32))
            for _ in range(n_sets)]
    with torch.cuda.stream(stream):
        for i in range(2 * n_sets):
            x, w, o = sets[i % n_sets]
            dg.conv2d_forward(x, w, o, p, code, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(calls):
            x, w, o = sets[i % n_sets]
            dg.conv2d_forward(x, w, o, p, code, stream)
        e1.record(stream)
    stream.synchronize()
    rc = dg.conv2d_grad_input_check_errors(stream)
    if rc != 0:
        raise RuntimeError(f"forward: {dg.conv2d_grad_input_status_string(rc)}")
    return e0.elapsed_time(e1) / calls


# The fused RMSNorm + matmul (include/rmsnorm_matmul.h): an LLM projection
# shape -- 8192 tokens, hidden size 4096, 4096 outputs -- in bf16.
RMS_SHAPE = {"m": 8192, "n": 4096, "k": 4096, "dtype": "bf16", "eps": 1e-6}


def rmsnorm_flops_bytes(m: int, n: int, k: int, esize: int = 2):
    """Useful FLOPs (2 m n k: the products; the norm adds O(m k)) and
    algorithmic bytes (X, W_norm and W_proj read once, C float32 written once)."""
    return 2.0 * m * n * k, float(m * k * esize + k * esize + k * n * esize + m * n * 4)


def rmsnorm_call(dg, dev, stream, calls=40):
    """The fused RMSNorm + matmul of RMS_SHAPE, back to back (its 224 MB of
    operands and result exceed L2, so every call streams from HBM), timed with
    events; returns (ms per call, kernel id)."""
    import torch
    sh = RMS_SHAPE
    m, n, k = sh["m"], sh["n"], sh["k"]
    gen = torch.Generator().manual_seed(0)
    x = (torch.randn(m, k, generator=gen) * torch.exp(torch.empty(m, 1).uniform_(-2.3, 2.3, generator=gen)))
    wn = torch.empty(k).uniform_(0.5, 1.5, generator=gen)
    wp = torch.randn(k, n, generator=gen) / math.sqrt(k)
    tdt = torch.bfloat16
    x, wn, wp = x.to(tdt).to(dev), wn.to(tdt).to(dev), wp.to(tdt).to(dev)
    c = torch.empty(m, n, device=dev)
    p = dg.RmsParams(m, n, k, sh["eps"])
    code = dg.DTYPE_CODE[sh["dtype"]]
    kernel = dg.rmsnorm_matmul_select_kernel(x, wn, wp, c, p, code)
    with torch.cuda.stream(stream):
        for _ in range(3):
            dg.rmsnorm_matmul(x, wn, wp, c, p, code, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(calls):
            dg.rmsnorm_matmul(x, wn, wp, c, p, code, stream)
        e1.record(stream)
    stream.synchronize()
    rc = dg.rmsnorm_matmul_check_errors(stream)
    if rc != 0:
        raise RuntimeError(f"rmsnorm_matmul: {dg.STATUS.get(rc, rc)}")
    return e0.elapsed_time(e1) / calls, kernel


# The attention gradient with respect to V (include/mha_grad_v.h): causal
# self-attention over 4096 positions, 32 query heads sharing 8 KV heads,
# head_dim 64, bf16.
MHA_SHAPE = {"q_seq": 4096, "kv_seq": 0, "num_heads": 32, "num_kv_heads": 8, "head_dim": 64,
             "window_size": 0, "dtype": "bf16"}


def mha_useful_flops(q_seq: int, kv_seq: int, num_heads: int, head_dim: int, window: int) -> float:
    """4 head_dim FLOPs (the score's dot product and the P dO update) for every
    (query, key, head) that the mask keeps: keys t < kv with t <= pos when
    causal (kv_seq == 0) and t > pos - window when window > 0."""
    import numpy as np
    kv = q_seq if kv_seq == 0 else kv_seq
    pos = np.arange(q_seq, dtype=np.int64)
    hi = np.minimum(pos if kv_seq == 0 else np.full_like(pos, kv - 1), kv - 1)
    lo = np.maximum(pos - window + 1, 0) if window > 0 else np.zeros_like(pos)
    pairs = int(np.maximum(hi - lo + 1, 0).sum())
    return 4.0 * head_dim * num_heads * pairs


def mha_call(dg, dev, stream, calls=20):
    """The attention dV of MHA_SHAPE back to back, timed with events; returns
    (ms per call, kernel id)."""
    import torch
    sh = MHA_SHAPE
    qs, nh, nkv, hd = sh["q_seq"], sh["num_heads"], sh["num_kv_heads"], sh["head_dim"]
    kv = qs if sh["kv_seq"] == 0 else sh["kv_seq"]
    gen = torch.Generator().manual_seed(0)
    q = torch.randn(qs, nh, hd, generator=gen).to(torch.bfloat16).to(dev)
    k = torch.randn(kv, nkv, hd, generator=gen).to(torch.bfloat16).to(dev)
    go = torch.randn(qs, nh, hd, generator=gen).to(torch.bfloat16).to(dev)
    # Forward statistics of a plausible size (they only set P's scale here; the
    # parity tests use exact ones): max = |q| |k| / sqrt(d) bound, log_sum = log(pos + 1).
    lse = torch.empty(qs, nh, 2, device=dev)
    lse[..., 0] = 4.0
    lse[..., 1] = torch.log(torch.arange(1, qs + 1, device=dev, dtype=torch.float32))[:, None]
    dv = torch.empty(kv, nkv, hd, device=dev)
    p = dg.MhaParams(qs, sh["kv_seq"], nh, nkv, hd, sh["window_size"])
    code = dg.DTYPE_CODE[sh["dtype"]]
    kernel = dg.mha_grad_v_select_kernel(q, k, go, lse, dv, p, code)
    with torch.cuda.stream(stream):
        for _ in range(3):
            dg.mha_grad_v(q, k, go, lse, dv, p, code, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(calls):
            dg.mha_grad_v(q, k, go, lse, dv, p, code, stream)
        e1.record(stream)
    stream.synchronize()
    rc = dg.mha_grad_v_check_errors(stream)
    if rc != 0:
        raise RuntimeError(f"mha_grad_v: {dg.STATUS.get(rc, rc)}")
    return e0.elapsed_time(e1) / calls, kernel


def run_gpu(args, wl, key):
    import torch
    import torch.distributed as dist

    import conv2d_backward_implicit_gb300 as dg
    from conv2d_backward_implicit_gb300 import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if dist_on:
        dist.init_process_group("nccl", device_id=dev)
    dg.library()

    # Data parallel over the batch: this rank's shard [lo, hi) of the global
    # batch of N x world images (its own seeded grad_out), the same weights on
    # every rank, its own grad_in slice; no exchange step.
    lo, hi = shard_bounds(wl.N * world, world, rank)
    assert hi - lo == wl.N
    g_cpu, _ = workloads.make_inputs(wl, seed=rank)
    _, w_cpu = workloads.make_inputs(wl, seed=0)
    p = dg.params_from_shapes(g_cpu.shape, w_cpu.shape, wl.H, wl.W, wl.stride, wl.padding_h,
                              wl.padding_w)
    code = dg.DTYPE_CODE[wl.dtype]
    kernel = dg.conv2d_grad_input_select_kernel(p, code)
    ws = dg.conv2d_grad_input_workspace_size(p, code)
    alg = algorithmic_bytes(wl)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 * 2**20)
    n_sets = max(2, math.ceil(3 * l2 / alg))
    sets = []
    for _ in range(n_sets):
        sets.append({"g": g_cpu.to(dev), "w": w_cpu.to(dev),
                     "out": torch.empty(wl.grad_in_shape, device=dev, dtype=torch.float32),
                     "packed": torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)})
    stream = torch.cuda.Stream(dev)

    def step(i, st, ev=None):
        s = sets[i % n_sets]
        if ws > 0:
            dg.conv2d_grad_input_pack_weight(s["w"], s["packed"], ws, p, code, st)
            if ev is not None:
                ev[0].record(st)
            dg.conv2d_grad_input_prepacked(s["g"], s["packed"], s["out"], p, code, st)
        else:
            if ev is not None:
                ev[0].record(st)
            dg.conv2d_grad_input_prepacked(s["g"], s["w"], s["out"], p, code, st)
        if ev is not None:
            ev[1].record(st)

    launches_per_step = 2 if ws > 0 else 1  # pack + dgrad, or dgrad alone
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i, stream)
    stream.synchronize()
    rc = dg.conv2d_grad_input_check_errors(stream)
    if rc != 0:
        raise RuntimeError(f"warm-up failed: {dg.conv2d_grad_input_status_string(rc)}")

    # Graph of one step per buffer set.  No event nodes inside: the pack and
    # dgrad kernels are launched with programmatic stream serialization, and an
    # event between two kernels would stop one's prologue overlapping the
    # other's tail.
    def make_graph(build):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            build()
        for _ in range(3):
            gr.replay()
        stream.synchronize()
        return gr

    step_graph = make_graph(lambda: [step(i, stream) for i in range(n_sets)])

    def main_only(i, st, ev=None):
        s = sets[i % n_sets]
        src = s["packed"] if ws > 0 else s["w"]
        if ev is not None:
            ev[0].record(st)
        dg.conv2d_grad_input_prepacked(s["g"], src, s["out"], p, code, st)
        if ev is not None:
            ev[1].record(st)

    if ws > 0:  # weights packed once per set for the kernel-only region
        for i in range(n_sets):
            s = sets[i]
            dg.conv2d_grad_input_pack_weight(s["w"], s["packed"], ws, p, code, stream)
    main_graph = make_graph(lambda: [main_only(i, stream) for i in range(n_sets)])

    K = args.steps
    reps, rest = divmod(K, n_sets)
    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local] \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else str(local)
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        gpu_id = "GPU-" + str(uuid) if not str(uuid).startswith("GPU-") else str(uuid)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    # The kernel-only region: at least 200 back-to-back launches whatever --steps is.
    main_reps = max(1, math.ceil(200 / n_sets))
    if dist_on:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        # Timed region 1: exactly K steps (pack + dgrad, or dgrad alone, each).
        ev[0].record(stream)
        for _ in range(reps):
            step_graph.replay()
        for i in range(rest):
            step(i, stream)
        ev[1].record(stream)
        # Timed region 2: back-to-back dgrad launches alone, for the kernel's
        # per-launch time (the roofline's denominator).
        ev[2].record(stream)
        for _ in range(main_reps):
            main_graph.replay()
        ev[3].record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    if dist_on:
        dist.barrier()
    sampler.mark(wall0, wall1)
    time.sleep(0.15)
    sampler.stop()
    rc = dg.conv2d_grad_input_check_errors(stream)
    if rc != 0:
        raise RuntimeError(f"timed region failed: {dg.conv2d_grad_input_status_string(rc)}")
    local_ms = ev[0].elapsed_time(ev[1])
    max_ms = reduce_max(local_ms, dist_on, dev)
    flops = useful_flops(wl)
    value = aggregate_throughput(flops, K, world, max_ms)
    k_ms = reduce_max(ev[2].elapsed_time(ev[3]), dist_on, dev) / (main_reps * n_sets)

    # For reference: one launch timed alone (event pair right around it, after a
    # sleep kernel so the queue is full), averaged over the buffer sets.
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(n_sets)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(50_000_000)
        for i in range(n_sets):
            main_only(i, stream, pairs[i])
    stream.synchronize()
    k_ms_isolated = statistics.mean(a.elapsed_time(b) for a, b in pairs)

    # End to end through the public one-call API with pinned host buffers:
    # every step copies its inputs host -> device, runs conv2d_grad_input and
    # copies grad_in back, all inside the timed region.  Steps are pipelined
    # over three streams (copy in, compute, copy out) and two device buffer
    # sets, so step i's copy-out overlaps step i+1's copy-in and kernel.
    g_host = g_cpu.pin_memory()
    w_host = w_cpu.pin_memory()
    out_hosts = [torch.empty(wl.grad_in_shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    bufs = [(sets[k]["g"], sets[k]["w"], sets[k]["out"]) for k in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_k = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    Ke = max(3, min(K, 200))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    for it in range(Ke + 3):
        k = it % 2
        gd, wd, od = bufs[k]
        if it == 3:
            e0.record(s_in)
        with torch.cuda.stream(s_in):
            if it >= 2:
                s_in.wait_event(ev_k[k])  # the kernel two steps back has read these inputs
            gd.copy_(g_host, non_blocking=True)
            wd.copy_(w_host, non_blocking=True)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if it >= 2:
            stream.wait_event(ev_out[k])  # grad_in of two steps back has been copied out
        dg.conv2d_grad_input(gd, wd, od, p, code, stream)
        ev_k[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_k[k])
            out_hosts[k].copy_(od, non_blocking=True)
            ev_out[k].record(s_out)
    s_out.wait_event(ev_out[(Ke + 2) % 2])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    rc = dg.conv2d_grad_input_check_errors(stream)
    if rc != 0:
        raise RuntimeError(f"e2e failed: {dg.conv2d_grad_input_status_string(rc)}")
    e2e_ms = reduce_max(e0.elapsed_time(e1), dist_on, dev)
    e2e_value = aggregate_throughput(flops, Ke, world, e2e_ms)
    out_host = out_hosts[0]

    peaks, peak_src = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    # fp32 inputs run on TF32 tensor cores: their peak is a TF32 matmul timed here.
    need_tf32 = wl.dtype == "f32" or (world == 1 and not args.no_per_config)
    tf32_peak = measure_tf32_peak(dev) if need_tf32 else None
    tf32_src = ("measured by bench.py on this GPU: torch.matmul float32 8192^3 with TF32 "
                "allowed, best of 10")

    def tc_peak_of(dtype):
        return (tf32_peak, tf32_src) if dtype == "f32" else (bf16_peak, peak_src)

    tc_peak, tc_src = tc_peak_of(wl.dtype)
    achieved_gbs = alg / (k_ms * 1e-3) / 1e9
    achieved_tflops = flops / (k_ms * 1e-3) / 1e12
    traffic = recorded_traffic(key)
    out = None
    if rank == 0:
        clocks = sampler.summary()
        out = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": max_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "f16": "f16", "f32": "tf32"}[wl.dtype] + " in, f32 accumulate/out",
            "data": "synthetic (seeded torch.Generator, recipe of the workload)",
            "config": dict(workload_config(
                wl, key, l2_note=f"rotating {n_sets} buffer sets of {alg / 1e6:.1f} MB "
                                 f"({n_sets * alg / 1e6:.0f} MB > 3x L2 {l2 / 1e6:.0f} MB)"),
                global_batch=wl.N * world, per_rank_batch=wl.N,
                parallelism=f"dp{world} (batch shards of {wl.N} images, weights replicated, "
                            "no collective)"),
            "kernel": {1: "tcgen05", 2: "cuda-core"}.get(kernel, str(kernel)),
            "gpu_launches": K * launches_per_step + main_reps * n_sets,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": achieved_gbs / hbm_peak,
                         "traffic": traffic,
                         "traffic_over_algorithmic": traffic / alg if traffic else None,
                         "kernel_ms": k_ms,
                         "kernel_ms_isolated": k_ms_isolated,
                         "kernel_timing": f"{main_reps * n_sets} back-to-back dgrad launches "
                                          "in the timed region (graph replay, events around it)",
                         "algorithmic_bytes": alg, "peak_source": peak_src},
            "tensor_roofline": {"achieved": achieved_tflops, "peak": tc_peak, "unit": "TFLOP/s",
                                "frac": achieved_tflops / tc_peak, "peak_source": tc_src},
            "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": g_cpu.numel() * g_cpu.element_size()
                    + w_cpu.numel() * w_cpu.element_size(),
                    "d2h_bytes_per_step": out_host.numel() * 4, "steps": Ke},
            "clocks": clocks,
        }
        if world == 1 and not args.no_per_config:
            # The metric is per workload: the dgrad kernel alone on each of the
            # five, same cold-L2 protocol (the bench workload's own line above).
            per = {}
            for other_key in ("tiny", "resnet", "strided", "pointwise", "stem"):
                owl = workloads.BY_KEY[other_key]
                o_ms, o_alg, o_kernel = kernel_only(dg, workloads, owl, other_key, dev, stream)
                o_peak, o_src = tc_peak_of(owl.dtype)
                o_gbs = o_alg / (o_ms * 1e-3) / 1e9
                o_tf = useful_flops(owl) / (o_ms * 1e-3) / 1e12
                o_traffic = recorded_traffic(other_key)
                per[other_key] = {"kernel_us": o_ms * 1e3, "tflops": o_tf,
                                  "hbm_frac": o_gbs / hbm_peak, "tensor_frac": o_tf / o_peak,
                                  "tensor_peak": o_peak, "dtype": owl.dtype,
                                  "kernel": {1: "tcgen05", 2: "cuda-core"}.get(o_kernel, str(o_kernel)),
                                  "traffic": o_traffic,
                                  "traffic_over_algorithmic": o_traffic / o_alg if o_traffic else None}
            out["per_config"] = per
            out["tf32_peak"] = {"value": tf32_peak, "unit": "TFLOP/s", "source": tf32_src}
            # The forward convolution of the bench layer, and of the strided
            # layer (stride 2: space-to-depth copy of x + weight split, then
            # the stride-1 path).
            f_ms = forward_call(dg, workloads, wl, dev, stream)
            out["forward"] = {"op": "conv2d_forward (weight flip + kernel, pack in the kernel or before it)",
                              "workload": wl.name, "ms_per_call": f_ms,
                              "tflops": useful_flops(wl) / (f_ms * 1e-3) / 1e12}
            if wl.stride == 1:
                swl = workloads.STRIDED
                fs_ms = forward_call(dg, workloads, swl, dev, stream)
                out["forward_strided"] = {
                    "op": "conv2d_forward at stride 2 (space-to-depth of x, weight split, stride-1 path)",
                    "workload": swl.name, "ms_per_call": fs_ms,
                    "tflops": useful_flops(swl) / (fs_ms * 1e-3) / 1e12}
            # The fused RMSNorm + matmul (a second operation of the library).
            r_ms, r_kernel = rmsnorm_call(dg, dev, stream)
            r_flops, r_bytes = rmsnorm_flops_bytes(RMS_SHAPE["m"], RMS_SHAPE["n"], RMS_SHAPE["k"])
            r_tf = r_flops / (r_ms * 1e-3) / 1e12
            sustained = float(peaks.get("bf16_tflops_sustained", bf16_peak))
            out["rmsnorm_matmul"] = {
                "op": "rmsnorm_matmul: C = RmsNorm(X, W_norm) x W_proj, norm fused (one pass over X)",
                "workload": "m={m} n={n} k={k} {dtype} in, f32 out, eps={eps}".format(**RMS_SHAPE),
                "kernel": {1: "tcgen05", 2: "cuda-core"}.get(r_kernel, str(r_kernel)),
                "us_per_call": r_ms * 1e3, "tflops": r_tf,
                "tensor_frac": r_tf / bf16_peak, "tensor_peak": bf16_peak,
                "tensor_frac_sustained": r_tf / sustained, "tensor_peak_sustained": sustained,
                "hbm_frac": r_bytes / (r_ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": r_bytes}
            # The attention gradient with respect to V (a third operation).
            m_ms, m_kernel = mha_call(dg, dev, stream)
            sh = MHA_SHAPE
            m_tf = mha_useful_flops(sh["q_seq"], sh["kv_seq"], sh["num_heads"], sh["head_dim"],
                                    sh["window_size"]) / (m_ms * 1e-3) / 1e12
            out["mha_grad_v"] = {
                "op": "mha_grad_v: dV of attention, P recomputed from the forward statistics",
                "workload": ("q_seq={q_seq} causal, heads {num_heads} over {num_kv_heads} KV heads, "
                             "head_dim {head_dim}, {dtype} in, f32 out").format(**sh),
                "kernel": {1: "tcgen05", 2: "cuda-core"}.get(m_kernel, str(m_kernel)),
                "us_per_call": m_ms * 1e3, "tflops": m_tf,
                "tensor_frac": m_tf / bf16_peak, "tensor_peak": bf16_peak}
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(wl)
        print(json.dumps(out), flush=True)
    if dist_on:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def ncu_traffic_command(key: str) -> str:
    """The ncu capture whose CSV --record-traffic reads (one pass: DRAM bytes
    and duration only; no cache flush between launches, so the counts are
    steady-state traffic; one GPU, a few launches, no clock control)."""
    return ("ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
            "--print-units base --cache-control none --clock-control none "
            f"-k regex:dgrad_tc_kernel -s 2 -c 6 --csv --log-file traffic_{key}.csv "
            f"python bench.py --config {key} --profile-launches 10")


def profile_run(args, wl, key):
    """Only the dgrad kernel, args.profile_launches times back to back over the
    rotating buffer sets (weights packed beforehand), for an ncu capture."""
    import torch
    import conv2d_backward_implicit_gb300 as dg
    from conv2d_backward_implicit_gb300 import workloads
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    g_cpu, w_cpu = workloads.make_inputs(wl, seed=0)
    p = dg.params_from_shapes(g_cpu.shape, w_cpu.shape, wl.H, wl.W, wl.stride, wl.padding_h,
                              wl.padding_w)
    code = dg.DTYPE_CODE[wl.dtype]
    ws = dg.conv2d_grad_input_workspace_size(p, code)
    alg = algorithmic_bytes(wl)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 * 2**20)
    n_sets = min(max(2, math.ceil(3 * l2 / alg)), 64)
    stream = torch.cuda.Stream(dev)
    sets = []
    for _ in range(n_sets):
        s = {"g": g_cpu.to(dev), "out": torch.empty(wl.grad_in_shape, device=dev)}
        if ws > 0:
            s["src"] = torch.empty(ws, dtype=torch.uint8, device=dev)
            dg.conv2d_grad_input_pack_weight(w_cpu.to(dev), s["src"], ws, p, code, stream)
        else:
            s["src"] = w_cpu.to(dev)
        sets.append(s)
    for i in range(args.profile_launches):
        s = sets[i % n_sets]
        dg.conv2d_grad_input_prepacked(s["g"], s["src"], s["out"], p, code, stream)
    stream.synchronize()
    rc = dg.conv2d_grad_input_check_errors(stream)
    if rc != 0:
        raise RuntimeError(f"profile launches failed: {dg.conv2d_grad_input_status_string(rc)}")
    print(json.dumps({"profile_launches": args.profile_launches, "workload": wl.name,
                      "buffer_sets": n_sets}), flush=True)
    return 0


def profile_rmsnorm(args):
    """Only the fused RMSNorm + matmul, args.profile_rmsnorm times back to back
    on an m x 4096 x 4096 bf16 problem (m = args.rmsnorm_m), for an ncu capture."""
    import torch
    import conv2d_backward_implicit_gb300 as dg
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    m, n, k = args.rmsnorm_m, RMS_SHAPE["n"], RMS_SHAPE["k"]
    gen = torch.Generator().manual_seed(0)
    x = torch.randn(m, k, generator=gen).to(torch.bfloat16).to(dev)
    wn = torch.empty(k).uniform_(0.5, 1.5, generator=gen).to(torch.bfloat16).to(dev)
    wp = (torch.randn(k, n, generator=gen) / math.sqrt(k)).to(torch.bfloat16).to(dev)
    c = torch.empty(m, n, device=dev)
    p = dg.RmsParams(m, n, k, RMS_SHAPE["eps"])
    for _ in range(args.profile_rmsnorm):
        dg.rmsnorm_matmul(x, wn, wp, c, p, dg.DGRAD_BF16)
    rc = dg.rmsnorm_matmul_check_errors()
    if rc != 0:
        raise RuntimeError(f"rmsnorm_matmul: {dg.STATUS.get(rc, rc)}")
    print(json.dumps({"profile_rmsnorm": args.profile_rmsnorm, "m": m, "n": n, "k": k}), flush=True)
    return 0


def profile_mha(args):
    """Only the attention dV of MHA_SHAPE, args.profile_mha times back to back
    (the inputs of mha_call), for an ncu capture."""
    import torch
    import conv2d_backward_implicit_gb300 as dg
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    ms, kernel = mha_call(dg, dev, stream, calls=args.profile_mha)
    print(json.dumps({"profile_mha": args.profile_mha, "kernel": kernel, **MHA_SHAPE}), flush=True)
    return 0


def record_traffic_file(args, wl, key):
    """Writes profiles/dgrad_tc_<key>.traffic.json from the CSV of ncu_traffic_command."""
    with open(args.record_traffic) as f:
        launches = traffic_from_ncu_csv(f.read())
    if not launches:
        raise SystemExit(f"no dgrad_tc_kernel launches with DRAM counters in {args.record_traffic}")
    rec = traffic_record(launches, wl, key, ncu_traffic_command(key))
    path = os.path.join(ROOT, "profiles", f"dgrad_tc_{key}.traffic.json")
    with open(path, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps({"written": os.path.relpath(path, ROOT),
                      "dram_bytes_per_launch": rec["dram_bytes_per_launch"],
                      "traffic_over_algorithmic": rec["traffic_over_algorithmic"]}))
    return 0


PROBES = {"mma": "mma_rate.cu", "tma": "tma_rate.cu", "tma_store": "tma_store_rate.cu"}


def run_probe(name: str) -> int:
    """Builds (nvcc, sm_103a) and runs one of the probes beside the package:
    tcgen05.mma issue rate per shape, TMA load and TMA store throughput per
    copy shape and number of issuing threads -- the device rates the kernels'
    design rests on.  Prints the probe's own report."""
    import shutil
    src = os.path.join(ROOT, "conv2d_backward_implicit_gb300", "probes", PROBES[name])
    out_dir = os.path.join(ROOT, "conv2d_backward_implicit_gb300", "_build", "probes")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, name)
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", src, "-o", exe],
                   check=True)
    return subprocess.run([exe]).returncode


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="resnet",
                    choices=["tiny", "resnet", "strided", "pointwise", "stem"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the kernel-only figures of the other workloads")
    ap.add_argument("--profile-launches", type=int, default=0, metavar="L",
                    help="only launch the dgrad kernel L times (for an ncu capture)")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="write profiles/dgrad_tc_<config>.traffic.json from an ncu CSV")
    ap.add_argument("--profile-rmsnorm", type=int, default=0, metavar="L",
                    help="only launch the fused RMSNorm + matmul L times on an m x 4096 x 4096 bf16 "
                         "problem (for an ncu capture; m from --rmsnorm-m)")
    ap.add_argument("--rmsnorm-m", type=int, default=2048, help="rows of X for --profile-rmsnorm")
    ap.add_argument("--profile-mha", type=int, default=0, metavar="L",
                    help="only launch the attention dV of the bench shape L times after 3 warm-up launches "
                         "(for an ncu capture)")
    ap.add_argument("--probe", choices=sorted(PROBES), default=None,
                    help="build and run a device-rate probe (tcgen05.mma, TMA loads or stores)")
    args = ap.parse_args(argv)
    if args.probe:
        return run_probe(args.probe)
    from conv2d_backward_implicit_gb300 import workloads
    wl = workloads.BY_KEY[args.config]
    if args.record_traffic:
        return record_traffic_file(args, wl, args.config)
    if args.profile_launches > 0:
        return profile_run(args, wl, args.config)
    if args.profile_rmsnorm > 0:
        return profile_rmsnorm(args)
    if args.profile_mha > 0:
        return profile_mha(args)
    if args.impl == "reference":
        args.steps = 10 if args.steps is None else args.steps
        args.warmup = 1 if args.warmup is None else args.warmup
        return run_reference(args, wl, args.config)
    args.steps = 60000 if args.steps is None else args.steps
    args.warmup = 100 if args.warmup is None else args.warmup
    if args.warmup < 3:
        args.warmup = 3
    return run_gpu(args, wl, args.config)


if __name__ == "__main__":
    sys.exit(main())
