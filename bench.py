#!/usr/bin/env python3
"""Benchmark of the packed K-quant matmul (gemm_quant) on one GB300.

Workload (one step): the Qwen3-0.6B decode GEMV set at m = 1 -- 28 layers,
each with the q/k/v projections (2048x1024, 1024x1024, 1024x1024, stored as
one contiguous 4096x1024 q4_K matrix because they share their input), o
(1024x2048), gate/up (3072x1024 each, one contiguous 6144x1024 matrix) and
down (1024x3072).  Every layer runs four dependent stages, each a q8_K
quantization of its f32 activation followed by a q4_K decode GEMV, in layer
order, exactly as a decode step would call them.  Weights are seeded
synthetic q4_K blocks (seed 1); activations are N(0,1).  The 247.7 MB weight
set is held twice and consecutive steps alternate copies, so every step reads
its weights from HBM (each copy is larger than the 129 MB L2).

Prints one JSON line (rank 0).  `value` is device time over K steps (CUDA
graph of the C-ABI calls, inputs resident); `e2e` adds the per-step host to
device copy of the activations and the device to host copy of the outputs;
`roofline` is the GEMV kernel's algorithmic bytes per launch over its
average launch time; `cpu_baseline` times the oracle on the host cores.
`--impl reference` times the oracle alone as the reference arm.
"""
import argparse
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

QK = 256
Q4K_BYTES = 144
Q8K_BYTES = 292

# (name, n, k) per layer; q/k/v and gate/up are contiguous row ranges
LAYER = [("qkv", 2048 + 1024 + 1024, 1024), ("o", 1024, 2048),
         ("gate_up", 3072 + 3072, 1024), ("down", 1024, 3072)]
N_LAYERS = 28
SEED = 1
WORKLOAD = "qwen3-0.6b decode GEMV set, q4_K, m=1, 28 layers x (qkv, o, gate_up, down)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="plm", choices=["plm", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def layer_bytes():
    return sum(n * (k // QK) * Q4K_BYTES for _, n, k in LAYER)


def step_algorithmic_bytes(m=1):
    """Bytes the path must move per step: q4_K weights, q8_K activations
    (written by the quantizer, read by the GEMV), f32 x in and y out."""
    tot = 0
    for _, n, k in LAYER:
        nb = k // QK
        w = n * nb * Q4K_BYTES
        xq = m * nb * Q8K_BYTES
        tot += w + xq + m * n * 4          # GEMV
        tot += m * k * 4 + xq              # quantize
    return tot * N_LAYERS


def gemv_bytes_per_step(m=1):
    return N_LAYERS * sum(n * (k // QK) * Q4K_BYTES + m * (k // QK) * Q8K_BYTES + m * n * 4
                          for _, n, k in LAYER)


def weights_per_step():
    return N_LAYERS * sum(n * k for _, n, k in LAYER)


# --------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- inputs

def build_inputs(torch, dev, copies=2):
    import gen
    nb_total = layer_bytes() * N_LAYERS
    wcopies = []
    host_w = np.empty(nb_total, dtype=np.uint8)
    off = 0
    for layer in range(N_LAYERS):
        for j, (_, n, k) in enumerate(LAYER):
            sz = n * (k // QK) * Q4K_BYTES
            gen.q4K_blocks(SEED, layer * len(LAYER) + j, n, k, out=host_w[off:off + sz].reshape(n, -1))
            off += sz
    for _ in range(copies):
        wcopies.append(torch.from_numpy(host_w).to(dev))
    xs, offs = [], []
    for layer in range(N_LAYERS):
        for j, (_, n, k) in enumerate(LAYER):
            xs.append(gen.normal_f32(SEED, 1000 + layer * len(LAYER) + j, 1, k))
    return host_w, wcopies, xs


class Plan:
    """Device buffers and the ordered list of (quantize, GEMV) calls."""

    def __init__(self, torch, dev, wcopies, xs, m=1):
        self.torch = torch
        self.m = m
        self.calls = []
        xtot = sum(x.size for x in xs)
        self.x_host = torch.empty(xtot, dtype=torch.float32).pin_memory()
        self.x_dev = torch.empty(xtot, dtype=torch.float32, device=dev)
        xq_tot = sum(x.size // QK * Q8K_BYTES for x in xs)
        self.xq = torch.empty(xq_tot, dtype=torch.uint8, device=dev)
        ytot = N_LAYERS * sum(n for _, n, _ in LAYER) * m
        self.y_dev = torch.empty(ytot, dtype=torch.float32, device=dev)
        self.y_host = torch.empty(ytot, dtype=torch.float32).pin_memory()
        xo = qo = yo = wo = 0
        idx = 0
        for layer in range(N_LAYERS):
            for (_, n, k) in LAYER:
                x = xs[idx]
                idx += 1
                self.x_host[xo:xo + x.size] = torch.from_numpy(x.ravel())
                nbq = x.size // QK * Q8K_BYTES
                self.calls.append(dict(xo=xo, qo=qo, yo=yo, wo=wo, n=n, k=k))
                xo += x.size
                qo += nbq
                yo += n * m
                wo += n * (k // QK) * Q4K_BYTES
        self.x_dev.copy_(self.x_host)
        self.wcopies = wcopies

    def ptrs(self, c, copy):
        return (self.x_dev.data_ptr() + 4 * c["xo"], self.xq.data_ptr() + c["qo"],
                self.y_dev.data_ptr() + 4 * c["yo"], self.wcopies[copy].data_ptr() + c["wo"])

    def run(self, q, copy, stream, quantize=True, gemv=True):
        for c in self.calls:
            xp, qp, yp, wp = self.ptrs(c, copy)
            if quantize:
                q.plm_quantize_q8K(xp, qp, self.m, c["k"], stream=stream)
            if gemv:
                q.plm_gemv_q4K(wp, qp, yp, self.m, c["n"], c["k"], stream=stream)


# --------------------------------------------------------------- oracle

def cpu_oracle_step(xs, host_w, layers, threads):
    import oracle
    oracle.set_threads(threads)
    off = 0
    idx = 0
    for layer in range(N_LAYERS):
        for (_, n, k) in LAYER:
            sz = n * (k // QK) * Q4K_BYTES
            if layer < layers:
                xq = oracle.quantize_q8K(xs[idx])
                oracle.gemm_q4K_f32(host_w[off:off + sz], xq, 1, n, k)
            off += sz
            idx += 1


def cpu_baseline(xs, host_w, budget_s=10.0):
    import oracle
    cores = len(os.sched_getaffinity(0))
    layer_bytes_alg = step_algorithmic_bytes() / N_LAYERS
    t0 = time.perf_counter()
    cpu_oracle_step(xs, host_w, 1, cores)           # warm (one layer)
    dt1 = time.perf_counter() - t0
    layers = max(1, min(N_LAYERS, int(budget_s / max(dt1, 1e-6) / 2)))
    reps = 0
    t0 = time.perf_counter()
    while True:
        cpu_oracle_step(xs, host_w, layers, cores)
        reps += 1
        el = time.perf_counter() - t0
        if el > budget_s / 2 or reps >= 50:
            break
    gbs = layer_bytes_alg * layers * reps / el / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "threads": oracle.max_threads(),
            "sample": "%d of 28 layers x %d passes (q8_K quantize + q4_K f32 oracle GEMV, "
                      "OpenMP over output rows), %.1f s" % (layers, reps, el)}


# --------------------------------------------------------------- main

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "plm" else "gloo")
        pg = dist
    return world, rank, local, pg


def run_reference(args, world, rank, pg):
    if rank != 0:
        return
    import gen  # noqa: F401
    host_w = np.empty(layer_bytes() * N_LAYERS, dtype=np.uint8)
    import gen as G
    off = 0
    for layer in range(N_LAYERS):
        for j, (_, n, k) in enumerate(LAYER):
            sz = n * (k // QK) * Q4K_BYTES
            G.q4K_blocks(SEED, layer * len(LAYER) + j, n, k, out=host_w[off:off + sz].reshape(n, -1))
            off += sz
    xs = [G.normal_f32(SEED, 1000 + i, 1, k) for i, (_, _, k) in
          enumerate([c for _ in range(N_LAYERS) for c in LAYER])]
    import oracle
    cores = len(os.sched_getaffinity(0))
    t0 = time.perf_counter()
    cpu_oracle_step(xs, host_w, 1, cores)
    per_layer = time.perf_counter() - t0
    layers = max(1, min(N_LAYERS, int(2.0 / max(per_layer, 1e-6))))
    for _ in range(args.warmup):
        cpu_oracle_step(xs, host_w, layers, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_oracle_step(xs, host_w, layers, cores)
    el = time.perf_counter() - t0
    alg = step_algorithmic_bytes() / N_LAYERS * layers
    val = alg * args.steps / el / 1e9
    sample = "%d of 28 layers per step (q8_K quantize + q4_K f32 oracle GEMV, OpenMP rows)" % layers
    print(json.dumps({
        "impl": "reference", "metric": "q4_K decode GEMV throughput (HBM GB/s of algorithmic bytes)",
        "value": val, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8xint4 -> f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "m": 1, "seed": SEED},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "threads": oracle.max_threads(), "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank, pg)
        return
    import torch
    import quant_packed_gemv_gb300 as q
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q.load()

    host_w, wcopies, xs = build_inputs(torch, dev)
    plan = Plan(torch, dev, wcopies, xs)
    stream = torch.cuda.Stream(device=dev)
    launches_per_step = 2 * len(plan.calls)

    # eager warm-up, then one CUDA graph per weight copy
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            plan.run(q, i % 2, stream)
    torch.cuda.synchronize()
    graphs, gemv_graphs = [], []
    for copy in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            plan.run(q, copy, stream)
        graphs.append(g)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            plan.run(q, copy, stream, quantize=False)
        gemv_graphs.append(g2)
    torch.cuda.synchronize()

    def barrier():
        if pg is not None:
            pg.barrier()

    def timed(fn, steps):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for s in range(steps):
            fn(s)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms = ev0.elapsed_time(ev1)
        if pg is not None:
            t = torch.tensor([ms], device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            ms = float(t.item())
        return ms

    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            graphs[s % 2].replay()
    sampler = ClockSampler(local)
    sampler.start()
    with torch.cuda.stream(stream):
        ms = timed(lambda s: graphs[s % 2].replay(), args.steps)
        gemv_ms = timed(lambda s: gemv_graphs[s % 2].replay(), args.steps)

        # end to end: host activations in, results out, every step
        h2d = plan.x_host.numel() * 4
        d2h = plan.y_host.numel() * 4

        def e2e_step(s):
            plan.x_dev.copy_(plan.x_host, non_blocking=True)
            graphs[s % 2].replay()
            plan.y_host.copy_(plan.y_dev, non_blocking=True)
        for s in range(2):
            e2e_step(s)
        t0 = time.perf_counter()
        e2e_ms = timed(e2e_step, args.steps)
        e2e_wall = (time.perf_counter() - t0) * 1e3
    clocks = sampler.stop()

    ms_step = ms / args.steps
    alg = step_algorithmic_bytes()
    value = world * alg / (ms_step * 1e-3) / 1e9
    gemv_launch_ms = gemv_ms / args.steps / len(plan.calls)
    gemv_alg_per_launch = gemv_bytes_per_step() / len(plan.calls)
    achieved = gemv_alg_per_launch / (gemv_launch_ms * 1e-3) / 1e9
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    e2e_value = world * alg / (max(e2e_ms, e2e_wall) / args.steps * 1e-3) / 1e9

    out = {
        "metric": "q4_K decode GEMV throughput (HBM GB/s of algorithmic bytes)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8xint4 -> f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "m": 1, "seed": SEED,
                   "weights_mb": layer_bytes() * N_LAYERS / 1e6,
                   "l2": "inputs larger than L2: two 247.7 MB weight copies, alternate steps",
                   "launch": "CUDA graph of the C-ABI calls, 4 dependent (quantize, GEMV) stages per layer"},
        "weights_per_s": world * weights_per_step() / (ms_step * 1e-3),
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "gemv_q4K_kernel<1>", "peak_source": peak_src,
                     "avg_launch_us": gemv_launch_ms * 1e3,
                     "bytes_per_launch": gemv_alg_per_launch},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": max(e2e_ms, e2e_wall) / args.steps},
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(xs, host_w)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
