"""Benchmark of the fused decode-GEMV over entropy-coded BF16 weights.

Workload (default): batch-1 y = W x for a 4096 x 4096 BF16 matrix W ~ N(0, 0.02), x ~ N(0, 1),
with 24 distinct device copies of the compressed matrix (about 540 MB, four times the 129 MB L2)
rotated so no launch reads from L2 what the previous one left there. One step = one GEMV over
every copy (24 launches, replayed as one CUDA graph). value = microseconds per matrix.

Also reported: the roofline of the GEMV kernel (algorithmic bytes per launch / average launch
time against the measured HBM copy bandwidth), the same shape through cuBLAS BF16 (torch.mv) with
the same rotation, an end-to-end figure through the public API with host buffers (x copied in,
y copied out every step), the SM clocks during the timed region, and the CPU oracle timed on the
host's cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl nwc|reference]
Multi-GPU: replicas only (the method has no exchange step); each rank runs the same workload on
its own GPU, the time is the max over ranks and value = that time / all matrices processed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused decode-GEMV µs/matrix & HBM GB/s (compressed) as % of GB300 peak"
N_ROWS = K_COLS = 4096
COPIES = 24
WORKLOAD = "square 4096x4096 BF16 batch-1 GEMV, 24 rotated copies"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_hash():
    h = hashlib.sha256()
    for f in ("kernels.cu", "nwc_format.h"):
        h.update(open(os.path.join(ROOT, "decode_gemv_nwc_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_key):
    """Per-launch DRAM bytes from an ncu capture recorded in profiles/traffic.txt
    ("<kernel hash> <workload key> <bytes per launch>"); None if the kernel changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    kh = kernel_hash()
    for line in open(p):
        parts = line.split("#")[0].split()
        if len(parts) == 3 and parts[0] == kh and parts[1] == workload_key:
            return int(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    def __init__(self, index):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
                vals = [v.strip() for v in out.stdout.strip().split(",")]
                if len(vals) == 6:
                    self.samples.append(vals)
            except Exception:
                pass
            self._stop.wait(0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[2 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


def dist_setup(gpus):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_sample(seconds_budget=12.0):
    """The CPU oracle as it stands: decode + FP64 matvec of one 4096x4096 blob per sample."""
    import oracle
    from decode_gemv_nwc_gb300 import synth
    w = synth.normal_bf16((N_ROWS, K_COLS), 0.02, seed=0)
    x = synth.activations_bf16(K_COLS, 1)
    blob = oracle.encode(w)
    times = []
    t_end = time.perf_counter() + seconds_budget
    while time.perf_counter() < t_end or not times:
        t0 = time.perf_counter()
        oracle.gemv(blob, x)
        times.append(time.perf_counter() - t0)
    return statistics.median(times) * 1e6, len(times)


def run_reference(args, rank, world):
    if rank != 0:
        return
    per = []
    for _ in range(args.warmup):
        oracle_sample(0.0)
    for _ in range(args.steps):
        us, _ = oracle_sample(0.0)
        per.append(us)
    v = statistics.mean(per)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "us/matrix", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "square 4096x4096 BF16 batch-1 GEMV (one matrix per step, CPU oracle)",
                   "matrix": [N_ROWS, K_COLS]},
        "cpu_baseline": {"value": v, "unit": "us/matrix", "cores": 1, "kind": "oracle",
                         "sample": "decode + FP64 matvec of one 4096x4096 blob per step"},
        "e2e": {"value": v, "unit": "us/matrix", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="nwc", choices=["nwc", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    import torch
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import decode_gemv_nwc_gb300 as nwc
    from decode_gemv_nwc_gb300 import build, synth
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())

    w = synth.normal_bf16((N_ROWS, K_COLS), 0.02, seed=0)
    x = synth.activations_bf16(K_COLS, 1)
    blob = nwc.encode(w)
    host = torch.from_numpy(np.frombuffer(blob, np.uint8).copy())
    mats = [nwc.Matrix(blob, device_blob=host.to(dev)) for _ in range(COPIES)]
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    ys = torch.empty((COPIES, N_ROWS), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # one step = one GEMV per copy, captured once as a CUDA graph
    with torch.cuda.stream(stream):
        for i, m in enumerate(mats):
            m.gemv(xd, y=ys[i], stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i, m in enumerate(mats):
            m.gemv(xd, y=ys[i], stream=stream)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    st, flags = nwc.check(stream)
    assert st == 0, f"device error word {flags:#x}"

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            ev1.record(stream)
        ev1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, world)
    launches = args.steps * COPIES
    us_per_matrix_job = ms * 1e3 / (launches * world)
    us_per_launch = ms_local * 1e3 / launches

    # algorithmic bytes per launch: the whole blob + x (BF16) + y (FP32)
    algo_bytes = len(blob) + 2 * K_COLS + 4 * N_ROWS
    peak, peak_kind = peaks()
    achieved = algo_bytes / (us_per_launch * 1e-6) / 1e9

    # cuBLAS BF16 matvec, same shape and rotation
    wd = torch.from_numpy(w.view(np.int16)).to(dev).view(torch.bfloat16)
    wcopies = [wd.clone() for _ in range(max(2, (512 << 20) // (2 * N_ROWS * K_COLS) + 1))]
    xb = xd.view(torch.bfloat16)
    yb = torch.empty((len(wcopies), N_ROWS), dtype=torch.bfloat16, device=dev)
    with torch.cuda.stream(stream):
        for i, wc in enumerate(wcopies):
            torch.mv(wc, xb, out=yb[i])
    stream.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        for i, wc in enumerate(wcopies):
            torch.mv(wc, xb, out=yb[i])
    for _ in range(3):
        g2.replay()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            g2.replay()
        ev1.record(stream)
    ev1.synchronize()
    cublas_us = ev0.elapsed_time(ev1) * 1e3 / (args.steps * len(wcopies))

    # end to end through the public API with host buffers
    x_pin = torch.from_numpy(x.view(np.int16)).pin_memory()
    y_pin = torch.empty((COPIES, N_ROWS), dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(xd)
    e2e_steps = max(3, args.steps // 2)

    def e2e_step():
        with torch.cuda.stream(stream):
            x_dev.copy_(x_pin, non_blocking=True)
            for i, m in enumerate(mats):
                m.gemv(x_dev, y=ys[i], stream=stream)
            y_pin.copy_(ys, non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        e2e_step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_us = e2e_s * 1e6 / (e2e_steps * COPIES * world)
    st, flags = nwc.check(stream)
    assert st == 0, f"device error word {flags:#x}"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        us, n = oracle_sample()
        cpu = {"value": us, "unit": "us/matrix", "cores": 1, "kind": "oracle",
               "sample": f"{n} runs of decode + FP64 matvec of one 4096x4096 blob (single-threaded C)"}

    traffic = recorded_traffic("square4096")
    if rank == 0:
        line = {
            "metric": METRIC, "value": us_per_matrix_job, "unit": "us/matrix", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "matrix": [N_ROWS, K_COLS], "weights": "bf16 entropy-coded",
                       "copies": COPIES, "blob_bytes": len(blob), "compressed_frac_of_bf16": len(blob) / (2 * N_ROWS * K_COLS),
                       "l2": f"inputs larger than L2: {COPIES} copies, {COPIES * len(blob) / 1e6:.0f} MB",
                       "graph": True, "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": traffic, "algorithmic_bytes_per_launch": algo_bytes,
                         "us_per_launch": us_per_launch},
            "decompressed_gbs": 2 * N_ROWS * K_COLS / (us_per_launch * 1e-6) / 1e9,
            "bf16_cublas": {"us_per_matrix": cublas_us, "gbs": 2 * N_ROWS * K_COLS / (cublas_us * 1e-6) / 1e9,
                            "speedup_of_nwc": cublas_us / us_per_launch},
            "e2e": {"value": e2e_us, "unit": "us/matrix", "h2d_bytes_per_step": 2 * K_COLS,
                    "d2h_bytes_per_step": 4 * N_ROWS * COPIES},
            "gpu_launches": launches,
            "clocks": clocks.summary(),
            "sm_count": nwc.sm_count(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
