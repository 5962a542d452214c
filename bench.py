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
    """SM clocks and throttle reasons from nvidia-smi's loop mode (every 20 ms, timestamped),
    read by a thread. start() returns once the first sample arrived (or after 5 s); summary()
    keeps the samples taken inside a wall-clock window (the timed region)."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.samples = []  # (epoch seconds, [sm, max, hw, hw_thermal, sw_thermal, sw_power])
        self.thread = None

    def _read(self):
        import datetime
        for line in self.proc.stdout:
            vals = [v.strip() for v in line.split(",")]
            if len(vals) != 7:
                continue
            try:
                ts = datetime.datetime.strptime(vals[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            self.samples.append((ts, vals[1:]))

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t_end = time.time() + 5.0
        while not self.samples and time.time() < t_end:
            time.sleep(0.01)
        return self

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except Exception:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [v for ts, v in self.samples if t0 - 0.005 <= ts <= t1 + 0.005]
        where = "timed region"
        if not inside and self.samples:  # region shorter than the interval: the nearest sample
            inside = [min(self.samples, key=lambda s: abs(s[0] - 0.5 * (t0 + t1)))[1]]
            where = "nearest sample"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(v[0]) for v in inside if v[0].replace(".", "").isdigit()]
        mx = [float(v[1]) for v in inside if v[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for v in inside for i in range(4) if v[2 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "interval_ms": self.INTERVAL_MS, "window": where}


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


def max_over_ranks(v, world, device="cuda"):
    """Max of a per-rank float over all ranks (the job's time is its slowest replica)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_matrix(max_ms, launches_per_rank, world):
    """Whole-job value: the slowest rank's time divided by the matrices all ranks processed."""
    return max_ms * 1e3 / (launches_per_rank * world)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_inputs():
    import oracle
    from decode_gemv_nwc_gb300 import synth
    w = synth.normal_bf16((N_ROWS, K_COLS), 0.02, seed=0)
    x = synth.activations_bf16(K_COLS, 1)
    return oracle.encode(w), x


def oracle_baseline(seconds_single=8.0, seconds_all=6.0):
    """The CPU oracle as it stands, on the host's cores: decode + FP64 matvec of the whole
    4096x4096 blob, (a) split by row blocks over every usable core (oracle.parallel: the same
    oracle library in spawned worker processes, results bit-identical to one process) and (b) in
    this process alone (one core). Each is the median over as many whole-matrix runs as fit its
    time budget (at least one)."""
    import oracle
    from oracle import parallel
    blob, x = oracle_inputs()

    def median_runs(fn, budget):
        times = []
        t_end = time.perf_counter() + budget
        while time.perf_counter() < t_end or not times:
            t0 = time.perf_counter()
            fn()
            times.append(time.perf_counter() - t0)
        return statistics.median(times) * 1e6, len(times)

    with parallel.Oracle(blob) as po:
        po.gemv(x)  # workers started and the blob paged in
        all_us, all_n = median_runs(lambda: po.gemv(x), seconds_all)
        cores = po.workers
    parallel.shutdown()
    one_us, one_n = median_runs(lambda: oracle.gemv(blob, x), seconds_single)
    return {"value": all_us, "unit": "us/matrix", "cores": cores, "kind": "oracle",
            "sample": f"{all_n} whole-matrix runs of decode + FP64 matvec of the 4096x4096 blob, rows split by "
                      f"8-row blocks over {cores} worker processes (one oracle each)",
            "single_core": {"value": one_us, "unit": "us/matrix", "cores": 1,
                            "sample": f"{one_n} whole-matrix runs in one process"}}


def time_graph(fn, stream, steps, warmup=3):
    """Captures fn() (launches on `stream`) once as a CUDA graph; returns ms per replay."""
    import torch
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / steps


def encode_on_host(w_dev, elem=0):
    """Device BF16 bits -> blob (the host encoder runs on the CPU cores)."""
    import decode_gemv_nwc_gb300 as nwc
    w = w_dev.cpu().numpy().view(np.uint16)
    return nwc.encode(w, elem=elem)


def extra_workloads(dev, stream, steps):
    """The other configurations of the pages' workloads, measured the same way."""
    import torch
    import decode_gemv_nwc_gb300 as nwc
    from decode_gemv_nwc_gb300 import synth
    out = {}
    peak, _ = peaks()

    # The odd shape of the square workload: 4095x4100 (a ragged last row block and column block),
    # 24 rotated copies as for the headline, then its decode; cuBLAS on the BF16 weights beside it.
    w = synth.normal_bf16((4095, 4100), 0.02, 1, device=dev)
    blob = encode_on_host(w)
    host = torch.from_numpy(np.frombuffer(blob, np.uint8).copy())
    omats = [nwc.Matrix(blob, device_blob=host.to(dev)) for _ in range(COPIES)]
    xo = torch.from_numpy(synth.activations_bf16(4100, 1001).view(np.int16)).to(dev)
    yo = torch.empty(4095, dtype=torch.float32, device=dev)
    odd_ms = time_graph(lambda: [m.gemv(xo, y=yo, stream=stream) for m in omats], stream, max(3, steps // 2))
    dec_o = [torch.empty((4095, 4100), dtype=torch.int16, device=dev) for _ in range(4)]
    odd_dec_ms = time_graph(lambda: [m.decode(out=dec_o[i % 4], stream=stream) for i, m in enumerate(omats)], stream,
                            max(3, steps // 10)) / COPIES
    wo = [w.view(torch.bfloat16).clone() for _ in range(COPIES)]
    ybo = torch.empty(4095, dtype=torch.bfloat16, device=dev)
    odd_bf16_ms = time_graph(lambda: [torch.mv(wc, xo.view(torch.bfloat16), out=ybo) for wc in wo], stream,
                             max(3, steps // 2))
    out["odd_4095x4100"] = {
        "workload": "4095x4100 BF16 batch-1 GEMV (ragged last row and column blocks), 24 rotated copies; decode",
        "us": odd_ms * 1e3 / COPIES, "compressed_bytes": len(blob),
        "frac_of_measured_hbm": (len(blob) + 2 * 4100 + 4 * 4095) / (odd_ms * 1e-3 / COPIES) / 1e9 / peak,
        "decode_us": odd_dec_ms * 1e3, "bf16_cublas_us": odd_bf16_ms * 1e3 / COPIES}
    del omats, wo, host, w, dec_o
    torch.cuda.empty_cache()

    # A small matrix of the stack (the k projection, 1024x2560: five blocks per SM, where the
    # launch's start-up and final sums weigh most); rotated copies beyond L2.
    kn, kk = 1024, 2560
    w = synth.normal_bf16((kn, kk), 0.02, 3, device=dev)
    blob = encode_on_host(w)
    kcopies = int(560e6 // len(blob)) + 1
    host = torch.from_numpy(np.frombuffer(blob, np.uint8).copy())
    kmats = [nwc.Matrix(blob, device_blob=host.to(dev)) for _ in range(kcopies)]
    xk = torch.from_numpy(synth.activations_bf16(kk, 1003).view(np.int16)).to(dev)
    yk = torch.empty(kn, dtype=torch.float32, device=dev)
    k_ms = time_graph(lambda: [m.gemv(xk, y=yk, stream=stream) for m in kmats], stream, max(3, steps // 10))
    wk = [w.view(torch.bfloat16).clone() for _ in range(kcopies)]
    ybk = torch.empty(kn, dtype=torch.bfloat16, device=dev)
    k_bf16_ms = time_graph(lambda: [torch.mv(wc, xk.view(torch.bfloat16), out=ybk) for wc in wk], stream,
                           max(3, steps // 10))
    route = {nwc.ROUTE_GEMV: "round-robin", nwc.ROUTE_LIST: "list"}[kmats[0].route()]
    out["k_proj_1024x2560"] = {
        "workload": f"1024x2560 BF16 batch-1 GEMV, {kcopies} rotated copies", "kernel": route,
        "us": k_ms * 1e3 / kcopies, "compressed_bytes": len(blob),
        "frac_of_measured_hbm": (len(blob) + 2 * kk + 4 * kn) / (k_ms * 1e-3 / kcopies) / 1e9 / peak,
        "bf16_cublas_us": k_bf16_ms * 1e3 / kcopies}
    del kmats, wk, host, w
    torch.cuda.empty_cache()

    # 36-layer decoder stack, one token = one GEMV per matrix (252), as one CUDA graph
    t0 = time.time()
    mats, xs, ys, wbf = [], {}, [], []
    comp_bytes = 0
    for layer in range(synth.N_LAYERS):
        for name, n, k in synth.LAYER_SHAPES:
            w = synth.layer_matrix(layer, name, device=dev)
            blob = encode_on_host(w)
            comp_bytes += len(blob)
            mats.append(nwc.Matrix(blob, device=dev))
            wbf.append(w.view(torch.bfloat16))
            if k not in xs:
                xs[k] = torch.from_numpy(synth.activations_bf16(k, 2000 + k).view(np.int16)).to(dev)
            ys.append(torch.empty(n, dtype=torch.float32, device=dev))
    build_s = time.time() - t0

    def stack():
        for m, y in zip(mats, ys):
            m.gemv(xs[m.k], y=y, stream=stream)

    yb = [torch.empty(w.shape[0], dtype=torch.bfloat16, device=dev) for w in wbf]

    def stack_bf16():
        for w, y in zip(wbf, yb):
            torch.mv(w, xs[w.shape[1]].view(torch.bfloat16), out=y)

    tok_ms = time_graph(stack, stream, max(3, steps // 2))
    tok_bf16 = time_graph(stack_bf16, stream, max(3, steps // 2))
    bf16_bytes = sum(2 * w.numel() for w in wbf)
    out["stack_token"] = {
        "workload": "36-layer stack (q,k,v,o,gate,up,down), one batch-1 GEMV per matrix, one CUDA graph",
        "gemvs": len(mats), "us_per_token": tok_ms * 1e3, "compressed_bytes": comp_bytes,
        "compressed_gbs": comp_bytes / (tok_ms * 1e-3) / 1e9, "frac_of_measured_hbm": comp_bytes / (tok_ms * 1e-3) / 1e9 / peak,
        "bf16_cublas_us_per_token": tok_bf16 * 1e3, "bf16_bytes": bf16_bytes, "speedup_vs_bf16": tok_bf16 / tok_ms,
        "build_seconds": build_s}
    del mats, wbf, ys, yb
    torch.cuda.empty_cache()

    # The same stack with fused projections (the NWC page's fuse step: q|k|v and gate|up share
    # their input, so each group is one matrix with its rows stacked): 144 GEMVs a token.
    t0 = time.time()
    mats, ys, wbf = [], [], []
    comp_bytes = 0
    for layer in range(synth.N_LAYERS):
        ws = {name: synth.layer_matrix(layer, name, device=dev) for name, _, _ in synth.LAYER_SHAPES}
        for group in (("q", "k", "v"), ("o",), ("gate", "up"), ("down",)):
            w = torch.cat([ws[g] for g in group]) if len(group) > 1 else ws[group[0]]
            blob = encode_on_host(w)
            comp_bytes += len(blob)
            mats.append(nwc.Matrix(blob, device=dev))
            wbf.append(w.view(torch.bfloat16))
            ys.append(torch.empty(w.shape[0], dtype=torch.float32, device=dev))
        del ws
    build_s = time.time() - t0
    yb = [torch.empty(w.shape[0], dtype=torch.bfloat16, device=dev) for w in wbf]
    tok_ms = time_graph(stack, stream, max(3, steps // 2))
    tok_bf16 = time_graph(stack_bf16, stream, max(3, steps // 2))
    out["stack_token_fused"] = {
        "workload": "36-layer stack with fused projections (q|k|v, o, gate|up, down), one CUDA graph",
        "gemvs": len(mats), "us_per_token": tok_ms * 1e3, "compressed_bytes": comp_bytes,
        "compressed_gbs": comp_bytes / (tok_ms * 1e-3) / 1e9, "frac_of_measured_hbm": comp_bytes / (tok_ms * 1e-3) / 1e9 / peak,
        "bf16_cublas_us_per_token": tok_bf16 * 1e3, "speedup_vs_bf16": tok_bf16 / tok_ms, "build_seconds": build_s}

    # The same chain with each launch bringing the next matrix's bytes into L2 (nwc_gemv_next):
    # a decoding step knows its sequence of matrices, so this keeps the model's ordering.
    def stack_next():
        for i, (m, y) in enumerate(zip(mats, ys)):
            m.gemv(xs[m.k], y=y, stream=stream, next=mats[i + 1] if i + 1 < len(mats) else None)

    nxt_ms = time_graph(stack_next, stream, max(3, steps // 2))
    out["stack_token_fused"]["us_per_token_with_next_prefetch"] = nxt_ms * 1e3
    out["stack_token_fused"]["speedup_vs_bf16_with_next_prefetch"] = tok_bf16 / nxt_ms

    # The same 144 products through nwc_gemv_list: one launch per layer (4 items) and one launch
    # for the whole token (144 items). The inputs here are independent synthetic vectors, as in
    # every stack line above; in a real decoding step each layer's products depend on the
    # previous ones through norms, attention and the activation, so only the per-layer form
    # keeps a model's ordering (its q|k|v, o, gate|up and down would still be four calls).
    list_items = [(m, xs[m.k], y) for m, y in zip(mats, ys)]

    def stack_list_layers():
        for i in range(0, len(list_items), 4):
            nwc.gemv_list(list_items[i:i + 4], stream=stream)

    lay_ms = time_graph(stack_list_layers, stream, max(3, steps // 2))
    all_ms = time_graph(lambda: nwc.gemv_list(list_items, stream=stream), stream, max(3, steps // 2))
    out["stack_token_fused_list"] = {
        "workload": "36-layer fused stack through nwc_gemv_list (independent inputs): one launch per layer, "
                    "and one launch for all 144 products",
        "us_per_token_layer_lists": lay_ms * 1e3, "us_per_token_one_list": all_ms * 1e3,
        "compressed_gbs_one_list": comp_bytes / (all_ms * 1e-3) / 1e9,
        "frac_of_measured_hbm_one_list": comp_bytes / (all_ms * 1e-3) / 1e9 / peak,
        "bf16_cublas_us_per_token": tok_bf16 * 1e3, "speedup_vs_bf16_one_list": tok_bf16 / all_ms,
        "speedup_vs_bf16_layer_lists": tok_bf16 / lay_ms}

    # Small-batch decoding on the fused stack: nb tokens per step through nwc_gemv_batch (each
    # weight decoded once for all nb vectors), against cuBLAS on the BF16 weights.
    xbat = {k: torch.from_numpy(np.stack([synth.activations_bf16(k, 3000 + k + v) for v in range(16)])
                                .view(np.int16)).to(dev) for k in {m.k for m in mats}}
    for nb in (2, 4, 8, 16):
        yB = [torch.empty((nb, m.n), dtype=torch.float32, device=dev) for m in mats]
        ybB = [torch.empty((nb, m.n), dtype=torch.bfloat16, device=dev) for m in mats]

        def stack_batch():
            for m, y in zip(mats, yB):
                m.gemv_batch(xbat[m.k][:nb], y=y, stream=stream)

        def stack_batch_bf16():
            for w, y in zip(wbf, ybB):
                torch.mm(xbat[w.shape[1]][:nb].view(torch.bfloat16), w.t(), out=y)
        b_ms = time_graph(stack_batch, stream, max(3, steps // 2))
        b_bf16 = time_graph(stack_batch_bf16, stream, max(3, steps // 2))
        out[f"stack_fused_batch{nb}"] = {
            "workload": f"36-layer fused stack, {nb} tokens per step (one fused GEMV per matrix for all {nb})",
            "us_per_step": b_ms * 1e3, "tokens_per_s": nb / (b_ms * 1e-3),
            "compressed_gbs": comp_bytes / (b_ms * 1e-3) / 1e9,
            "frac_of_measured_hbm": comp_bytes / (b_ms * 1e-3) / 1e9 / peak,
            "bf16_cublas_us_per_step": b_bf16 * 1e3, "speedup_vs_bf16": b_bf16 / b_ms}
        del yB, ybB
    del mats, wbf, ys, yb, xbat
    torch.cuda.empty_cache()

    # tied embedding / lm_head 151936 x 2560: gather 4096 ids, then the lm_head GEMV
    w = synth.normal_bf16((synth.VOCAB, synth.HIDDEN), 0.02, 7, device=dev)
    blob = encode_on_host(w)
    m = nwc.Matrix(blob, device=dev)
    x = torch.from_numpy(synth.activations_bf16(synth.HIDDEN, 9).view(np.int16)).to(dev)
    y = torch.empty(synth.VOCAB, dtype=torch.float32, device=dev)
    ids = torch.from_numpy(synth.token_ids(4096, synth.VOCAB, seed=8)).to(dev)
    g_out = torch.empty((4096, synth.HIDDEN), dtype=torch.int16, device=dev)
    lm_ms = time_graph(lambda: m.gemv(x, y=y, stream=stream), stream, steps)
    ga_ms = time_graph(lambda: m.gather(ids, out=g_out, stream=stream), stream, steps)
    wb = w.view(torch.bfloat16)
    yb = torch.empty(synth.VOCAB, dtype=torch.bfloat16, device=dev)
    lm_bf16 = time_graph(lambda: torch.mv(wb, x.view(torch.bfloat16), out=yb), stream, steps)
    out["lm_head"] = {"workload": "lm_head GEMV 151936x2560", "us": lm_ms * 1e3, "compressed_bytes": len(blob),
                      "compressed_gbs": len(blob) / (lm_ms * 1e-3) / 1e9,
                      "frac_of_measured_hbm": len(blob) / (lm_ms * 1e-3) / 1e9 / peak,
                      "bf16_cublas_us": lm_bf16 * 1e3, "speedup_vs_bf16": lm_bf16 / lm_ms}
    out["gather"] = {"workload": "gather 4096 ids from the 151936x2560 table", "us": ga_ms * 1e3,
                     "rows_per_s": 4096 / (ga_ms * 1e-3), "out_gbs": 4096 * synth.HIDDEN * 2 / (ga_ms * 1e-3) / 1e9}
    del m, w, wb
    torch.cuda.empty_cache()

    # fp8 gate 9728x2560 and down 2560x9728, 12 rotated copies each (> L2)
    for name, (n, k) in (("gate", (9728, 2560)), ("down", (2560, 9728))):
        w = synth.normal_bf16((n, k), 0.02, 50 + n, device=dev)
        blob = encode_on_host(w, elem=1)
        host = torch.from_numpy(np.frombuffer(blob, np.uint8).copy())
        ms8 = [nwc.Matrix(blob, device_blob=host.to(dev)) for _ in range(12)]
        x = torch.from_numpy(synth.activations_bf16(k, 77).view(np.int16)).to(dev)
        y = torch.empty(n, dtype=torch.float32, device=dev)

        def run8():
            for mm in ms8:
                mm.gemv(x, y=y, stream=stream)
        t = time_graph(run8, stream, steps) / len(ms8)
        wbs = [w.view(torch.bfloat16).clone() for _ in range(12)]
        yb = torch.empty(n, dtype=torch.bfloat16, device=dev)

        def runbf():
            for ww in wbs:
                torch.mv(ww, x.view(torch.bfloat16), out=yb)
        tb = time_graph(runbf, stream, steps) / len(wbs)
        out[f"fp8_{name}"] = {"workload": f"fp8 e4m3 {name} {n}x{k}, 12 rotated copies", "us": t * 1e3,
                              "compressed_bytes": len(blob), "fp8_bytes": n * k,
                              "compressed_gbs": len(blob) / (t * 1e-3) / 1e9,
                              "frac_of_measured_hbm": len(blob) / (t * 1e-3) / 1e9 / peak,
                              "bf16_cublas_us": tb * 1e3}
        del ms8, wbs
    torch.cuda.empty_cache()
    return out


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is one whole 4096x4096 matrix (decode +
    FP64 matvec), its rows split by 8-row blocks over every usable host core (oracle.parallel).
    value = mean step time, so the line reports exactly what it timed."""
    if rank != 0:
        return
    from oracle import parallel
    blob, x = oracle_inputs()
    with parallel.Oracle(blob) as po:
        for _ in range(args.warmup):
            po.gemv(x)
        per = []
        t_all = time.perf_counter()
        for _ in range(args.steps):
            t0 = time.perf_counter()
            po.gemv(x)
            per.append((time.perf_counter() - t0) * 1e6)
        wall = time.perf_counter() - t_all
        cores = po.workers
    parallel.shutdown()
    v = statistics.mean(per)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "us/matrix", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "matrix": [N_ROWS, K_COLS]},
        "cpu_baseline": {"value": v, "unit": "us/matrix", "cores": cores, "kind": "oracle",
                         "sample": f"per step: decode + FP64 matvec of the whole 4096x4096 blob, rows split by "
                                   f"8-row blocks over {cores} worker processes"},
        "timed_seconds": wall,
        "e2e": {"value": v, "unit": "us/matrix", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_batch_only(args):
    """Small-batch GEMV alone on the headline matrix (24 rotated copies, nb vectors): one JSON
    line, not the benchmark contract's; used for profiling the batch kernel."""
    import torch
    import decode_gemv_nwc_gb300 as nwc
    from decode_gemv_nwc_gb300 import build, synth
    build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    nb = args.only_batch
    w = synth.normal_bf16((N_ROWS, K_COLS), 0.02, seed=0)
    blob = nwc.encode(w)
    host = torch.from_numpy(np.frombuffer(blob, np.uint8).copy())
    mats = [nwc.Matrix(blob, device_blob=host.to(dev)) for _ in range(COPIES)]
    X = torch.from_numpy(np.stack([synth.activations_bf16(K_COLS, 1 + v) for v in range(nb)]).view(np.int16)).to(dev)
    Y = torch.empty((nb, N_ROWS), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    ms = time_graph(lambda: [m.gemv_batch(X, y=Y, stream=stream) for m in mats], stream, args.steps, args.warmup)
    st, flags = nwc.check(stream)
    assert st == 0, f"device error word {flags:#x}"
    us = ms * 1e3 / COPIES
    peak, peak_kind = peaks()
    algo = len(blob) + 2 * K_COLS * nb + 4 * N_ROWS * nb
    print(json.dumps({"workload": f"square {N_ROWS}x{K_COLS} BF16, {nb} vectors per GEMV, {COPIES} rotated copies",
                      "nb": nb, "us_per_matrix": us, "us_per_matrix_vector": us / nb,
                      "achieved_gbs": algo / (us * 1e-6) / 1e9, "frac_of_hbm": algo / (us * 1e-6) / 1e9 / peak,
                      "peak_kind": peak_kind, "gpu_launches": args.steps * COPIES}))


def run_only(args):
    """One workload of the pages' configurations alone (few launches, for profiling): the
    lm_head GEMV of the 151936x2560 table, the gather of 4096 ids from it, the fp8 gate / down
    GEMV (12 rotated copies), the odd 4095x4100 BF16 GEMV (24 rotated copies), the 24 rotated
    4096x4096 copies as one nwc_gemv_list launch, or the 1024x2560 GEMV (rotated copies beyond
    L2). One JSON line, not the benchmark contract's."""
    import torch
    import decode_gemv_nwc_gb300 as nwc
    from decode_gemv_nwc_gb300 import build, synth
    build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    peak, peak_kind = peaks()
    name = args.only
    if name in ("lm_head", "gather"):
        w = synth.normal_bf16((synth.VOCAB, synth.HIDDEN), 0.02, 7, device=dev)
        blob = encode_on_host(w)
        del w
        m = nwc.Matrix(blob, device=dev)
        if name == "lm_head":
            x = torch.from_numpy(synth.activations_bf16(synth.HIDDEN, 9).view(np.int16)).to(dev)
            y = torch.empty(synth.VOCAB, dtype=torch.float32, device=dev)
            ms = time_graph(lambda: m.gemv(x, y=y, stream=stream), stream, args.steps, args.warmup)
            gbs = len(blob) / (ms * 1e-3) / 1e9
            out = {"workload": "lm_head GEMV 151936x2560", "us": ms * 1e3, "compressed_gbs": gbs,
                   "frac_of_hbm": gbs / peak}
        else:
            ids = torch.from_numpy(synth.token_ids(4096, synth.VOCAB, seed=8)).to(dev)
            g = torch.empty((4096, synth.HIDDEN), dtype=torch.int16, device=dev)
            ms = time_graph(lambda: m.gather(ids, out=g, stream=stream), stream, args.steps, args.warmup)
            out = {"workload": "gather 4096 ids from the 151936x2560 table", "us": ms * 1e3,
                   "rows_per_s": 4096 / (ms * 1e-3)}
    elif name == "list4096":
        w = synth.normal_bf16((N_ROWS, K_COLS), 0.02, seed=0)
        blob = nwc.encode(w)
        host = torch.from_numpy(np.frombuffer(blob, np.uint8).copy())
        mats = [nwc.Matrix(blob, device_blob=host.to(dev)) for _ in range(COPIES)]
        x = torch.from_numpy(synth.activations_bf16(K_COLS, 1).view(np.int16)).to(dev)
        ys = torch.empty((COPIES, N_ROWS), dtype=torch.float32, device=dev)
        items = [(mm, x, ys[i]) for i, mm in enumerate(mats)]
        ms = time_graph(lambda: nwc.gemv_list(items, stream=stream), stream, args.steps, args.warmup) / COPIES
        gbs = len(blob) / (ms * 1e-3) / 1e9
        out = {"workload": "24 rotated 4096x4096 copies as one nwc_gemv_list launch", "us_per_matrix": ms * 1e3,
               "compressed_gbs": gbs, "frac_of_hbm": gbs / peak}
    elif name == "kproj":
        w = synth.normal_bf16((1024, 2560), 0.02, 3, device=dev)
        blob = encode_on_host(w)
        host = torch.from_numpy(np.frombuffer(blob, np.uint8).copy())
        mats = [nwc.Matrix(blob, device_blob=host.to(dev)) for _ in range(int(560e6 // len(blob)) + 1)]
        x = torch.from_numpy(synth.activations_bf16(2560, 1003).view(np.int16)).to(dev)
        y = torch.empty(1024, dtype=torch.float32, device=dev)
        ms = time_graph(lambda: [mm.gemv(x, y=y, stream=stream) for mm in mats], stream, args.steps,
                        args.warmup) / len(mats)
        gbs = len(blob) / (ms * 1e-3) / 1e9
        out = {"workload": f"1024x2560 BF16 GEMV, {len(mats)} rotated copies", "us": ms * 1e3,
               "compressed_gbs": gbs, "frac_of_hbm": gbs / peak, "route": mats[0].route()}
    elif name == "odd":
        w = synth.normal_bf16((4095, 4100), 0.02, 1, device=dev)
        blob = encode_on_host(w)
        host = torch.from_numpy(np.frombuffer(blob, np.uint8).copy())
        mats = [nwc.Matrix(blob, device_blob=host.to(dev)) for _ in range(COPIES)]
        x = torch.from_numpy(synth.activations_bf16(4100, 1001).view(np.int16)).to(dev)
        y = torch.empty(4095, dtype=torch.float32, device=dev)
        ms = time_graph(lambda: [mm.gemv(x, y=y, stream=stream) for mm in mats], stream, args.steps,
                        args.warmup) / len(mats)
        gbs = len(blob) / (ms * 1e-3) / 1e9
        out = {"workload": "4095x4100 BF16 GEMV, 24 rotated copies", "us": ms * 1e3, "compressed_gbs": gbs,
               "frac_of_hbm": gbs / peak}
    else:
        n, k = (9728, 2560) if name == "fp8_gate" else (2560, 9728)
        w = synth.normal_bf16((n, k), 0.02, 50 + n, device=dev)
        blob = encode_on_host(w, elem=1)
        host = torch.from_numpy(np.frombuffer(blob, np.uint8).copy())
        mats = [nwc.Matrix(blob, device_blob=host.to(dev)) for _ in range(12)]
        x = torch.from_numpy(synth.activations_bf16(k, 77).view(np.int16)).to(dev)
        y = torch.empty(n, dtype=torch.float32, device=dev)
        ms = time_graph(lambda: [mm.gemv(x, y=y, stream=stream) for mm in mats], stream, args.steps,
                        args.warmup) / len(mats)
        gbs = len(blob) / (ms * 1e-3) / 1e9
        out = {"workload": f"fp8 e4m3 {name[4:]} {n}x{k}, 12 rotated copies", "us": ms * 1e3,
               "compressed_gbs": gbs, "frac_of_hbm": gbs / peak}
    st, flags = nwc.check(stream)
    assert st == 0, f"device error word {flags:#x}"
    out["peak_kind"] = peak_kind
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="nwc", choices=["nwc", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--only-batch", type=int, default=0, metavar="NB",
                    help="time only nwc_gemv_batch with NB vectors on the headline matrix")
    ap.add_argument("--only", choices=["lm_head", "gather", "fp8_gate", "fp8_down", "odd", "list4096", "kproj"],
                    help="time only this workload (few launches; for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.only_batch:
        run_batch_only(args)
        return
    if args.only:
        run_only(args)
        return

    if args.impl == "reference":
        # the CPU oracle: rank 0 alone runs it (no GPU, no process group); other ranks exit
        run_reference(args, int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")))
        return

    import torch
    rank, world, local = dist_setup(args.gpus)

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
    clocks = ClockSampler(local).start()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    st, flags = nwc.check(stream)
    assert st == 0, f"device error word {flags:#x}"

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_on = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    t_off = time.time()
    time.sleep(2.5 * ClockSampler.INTERVAL_MS / 1000)  # the sample covering the region's end
    clocks.stop()
    torch.cuda.synchronize()
    barrier(world)
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, world)
    launches = args.steps * COPIES
    us_per_matrix_job = job_us_per_matrix(ms, launches, world)
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

    # One step: x from pinned host memory to the device, the GEMV over every copy, all y back to
    # pinned host memory, then the host waits for the step. The step's calls are captured once
    # as a CUDA graph (copies included) and replayed, as a serving loop would.
    def e2e_body():
        x_dev.copy_(x_pin, non_blocking=True)
        for i, m in enumerate(mats):
            m.gemv(x_dev, y=ys[i], stream=stream)
        y_pin.copy_(ys, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_body()
    stream.synchronize()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        e2e_body()

    def e2e_step():
        with torch.cuda.stream(stream):
            g_e2e.replay()
        stream.synchronize()

    for _ in range(2):
        e2e_step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_us = e2e_s * 1e6 / (e2e_steps * COPIES * world)
    assert torch.equal(y_pin, ys.cpu()), "the last step's results did not reach the host"
    st, flags = nwc.check(stream)
    assert st == 0, f"device error word {flags:#x}"

    # decode to BF16 (dequantization): every copy once per step into four rotated outputs, so that
    # neither the blobs nor the 33.5 MB outputs are read from L2 (reads blob bytes, writes 2NK bytes)
    dec_outs = [torch.empty((N_ROWS, K_COLS), dtype=torch.int16, device=dev) for _ in range(4)]
    dec_ms = time_graph(lambda: [m.decode(out=dec_outs[i % 4], stream=stream) for i, m in enumerate(mats)], stream,
                        max(3, args.steps // 10)) / COPIES
    extras = {"decode": {"workload": "decode 4096x4096 to BF16, 24 rotated copies into 4 rotated outputs",
                         "us": dec_ms * 1e3, "write_gbs": 2 * N_ROWS * K_COLS / (dec_ms * 1e-3) / 1e9,
                         "read_write_gbs": (len(blob) + 2 * N_ROWS * K_COLS) / (dec_ms * 1e-3) / 1e9,
                         "frac_of_measured_hbm": (len(blob) + 2 * N_ROWS * K_COLS) / (dec_ms * 1e-3) / 1e9 / peaks()[0]}}
    del dec_outs
    # The 24 copies' products as one nwc_gemv_list launch: no per-launch start-up or final sums
    # between matrices, so this is the decoder's steady-state rate on this shape (not the
    # headline, which is one matrix per launch).
    ys_list = torch.empty_like(ys)
    lst_ms = time_graph(lambda: nwc.gemv_list([(m, xd, ys_list[i]) for i, m in enumerate(mats)], stream=stream),
                        stream, args.steps)
    torch.cuda.synchronize()
    assert torch.equal(ys_list.view(torch.int32), ys.view(torch.int32)), "list launch differs from nwc_gemv"
    lst_us = lst_ms * 1e3 / COPIES
    extras["square4096_one_list"] = {
        "workload": "the 24 rotated 4096x4096 copies as one nwc_gemv_list launch", "us_per_matrix": lst_us,
        "achieved_gbs": algo_bytes / (lst_us * 1e-6) / 1e9, "frac_of_measured_hbm": algo_bytes / (lst_us * 1e-6) / 1e9 / peak,
        "speedup_vs_bf16_cublas": cublas_us / lst_us}
    del mats[1:]
    torch.cuda.empty_cache()
    if not args.quick:
        extras.update(extra_workloads(dev, stream, args.steps))
    st, flags = nwc.check(stream)
    assert st == 0, f"device error word {flags:#x}"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline()

    traffic = recorded_traffic("square4096")
    clk = clocks.summary(t_on, t_off)
    # the pages' decoder metric: SM clocks spent per 64 decoded weights, all SMs together
    f_sm = (clk.get("sm_mhz") or clk.get("sm_max_mhz") or 0) * 1e6
    clocks_per_64w = us_per_launch * 1e-6 * f_sm * nwc.sm_count() / (N_ROWS * K_COLS / 64) if f_sm else None
    if f_sm:
        extras["square4096_one_list"]["sm_clocks_per_64_weights"] = (
            extras["square4096_one_list"]["us_per_matrix"] * 1e-6 * f_sm * nwc.sm_count() / (N_ROWS * K_COLS / 64))
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
                         "frac_of_nominal_7900": achieved / 7900.0,
                         "traffic": traffic, "algorithmic_bytes_per_launch": algo_bytes,
                         "us_per_launch": us_per_launch},
            "decompressed_gbs": 2 * N_ROWS * K_COLS / (us_per_launch * 1e-6) / 1e9,
            "sm_clocks_per_64_weights": clocks_per_64w,
            "bf16_cublas": {"us_per_matrix": cublas_us, "gbs": 2 * N_ROWS * K_COLS / (cublas_us * 1e-6) / 1e9,
                            "speedup_of_nwc": cublas_us / us_per_launch},
            "e2e": {"value": e2e_us, "unit": "us/matrix", "h2d_bytes_per_step": 2 * K_COLS,
                    "d2h_bytes_per_step": 4 * N_ROWS * COPIES},
            "gpu_launches": launches,
            "clocks": clk,
            "sm_count": nwc.sm_count(),
            "cpu_baseline": cpu,
            "workloads": extras,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
