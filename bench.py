#!/usr/bin/env python3
"""Benchmark of the packed K-quant matmul (gemm_quant) on one GB300.

Workload of one step: the Qwen3-0.6B decode GEMV set at m = 1.  Each of the
28 layers holds seven distinct q4_K matrices (n x k): q 2048x1024,
k 1024x1024, v 1024x1024, o 1024x2048, gate 3072x1024, up 3072x1024,
down 1024x3072, laid out contiguously (247.7 MB).  Every matrix gets its own
f32 activation row (N(0,1), seed 1).  A step is one launch of the fused
producer + grouped GEMV (plm_quantize_gemv_q4K_grouped): each CTA quantizes
the f32 activations of its problems to q8_K in shared memory, then streams
its share of the 196 matrices' weight blocks.  The weight set is held twice
and consecutive steps alternate copies; each copy is larger than the 129 MB
L2, so weights come from HBM.  The K timed steps replay as one CUDA graph,
launched with plm_set_overlap(--overlap, default 2): each kernel is
scheduled while the one before it drains and starts copying its weights
(which nothing writes) before it waits for that kernel; activations are
read only after the wait.

Reported beside it (same JSON line):
  roofline      the fused kernel: algorithmic bytes per launch (weights,
                f32 activations, y) over its average launch time (CUDA
                events on its stream).
  decode_set_two_launch  the same step as two launches (plm_quantize_q8K
                over all 196 rows, then plm_gemv_q4K_grouped), with the
                GEMV's own roofline.
  decode_chain  the same layers run as a decoder must run them: per layer
                four dependent stages (qkv as one 4096-row matrix, o,
                gate/up as one 6144-row matrix, down), each a quantize and a
                single GEMV launch, in a CUDA graph.  Latency-bound.
  e2e           the step through the C ABI with the activations copied in
                from pinned host memory and the outputs copied back, the
                copies of one step overlapping the compute of the next on a
                second stream (and, as `serial`, without overlap; as
                `zero_copy`, the fused launch reading x from and writing y to
                pinned host memory itself, over the coherent CPU-GPU link).
  decode_chain_fused  the chain with one fused quantize + GEMV launch per
                stage.
  cpu_baseline  the oracle on the host cores, on a bounded sample.

`--impl reference` times the oracle alone (the reference arm).
`--case KIND FMT N K --m ...` times one entry point on one shape.
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
Q6K_BYTES = 210
Q5K_BYTES = 176
FMT_BYTES = {"q2K": 84, "q3K": 110, "q4K": Q4K_BYTES, "q5K": Q5K_BYTES, "q6K": Q6K_BYTES}
Q8K_BYTES = 292

# (name, n, k) of the seven matrices of one layer, in storage order
MATS = [("q", 2048, 1024), ("k", 1024, 1024), ("v", 1024, 1024), ("o", 1024, 2048),
        ("gate", 3072, 1024), ("up", 3072, 1024), ("down", 1024, 3072)]
# dependent stages of a decode layer: (first matrix, number of matrices fused by rows)
CHAIN = [(0, 3), (3, 1), (4, 2), (6, 1)]
N_LAYERS = 28
SEED = 1
WORKLOAD = ("qwen3-0.6b decode GEMV set: 28 layers x 7 q4_K matrices "
            "(q 2048x1024, k/v 1024x1024, o 1024x2048, gate/up 3072x1024, down 1024x3072), m=1")
METRIC = "q4_K decode GEMV throughput (HBM GB/s of algorithmic bytes)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="plm", choices=["plm", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", nargs=4, metavar=("KIND", "FMT", "N", "K"), default=None,
                    help="time one entry point alone, e.g. --case gemv q6K 151936 2048 "
                         "(KIND: gemv, gemv_x16, gemm, gemm_ws)")
    ap.add_argument("--m", type=int, nargs="+", default=[1],
                    help="activation rows for --case (several values: a sweep)")
    ap.add_argument("--no-chain", action="store_true",
                    help="skip the dependent per-layer decode chain measurement")
    ap.add_argument("--no-two-launch", action="store_true",
                    help="skip the two-launch (quantize, then grouped GEMV) comparison of the step")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the prefill GEMM, q6_K head and m-sweep measurements")
    ap.add_argument("--overlap", type=int, default=2, choices=[0, 1, 2],
                    help="plm_set_overlap mode: 0 plain stream order, 1 early launch, "
                         "2 early launch with weight prefetch (the weights here are never written)")
    return ap.parse_args()


def mat_list():
    """(layer, j, n, k, byte offset) of all 196 matrices in storage order."""
    out, off = [], 0
    for layer in range(N_LAYERS):
        for j, (_, n, k) in enumerate(MATS):
            out.append((layer, j, n, k, off))
            off += n * (k // QK) * Q4K_BYTES
    return out, off


def gemv_bytes(n, k, m=1):
    nb = k // QK
    return n * nb * Q4K_BYTES + m * nb * Q8K_BYTES + m * n * 4


def quant_bytes(k, m=1):
    return m * k * 4 + m * (k // QK) * Q8K_BYTES


def step_bytes(mats):
    """Two-launch step: the quantizer (f32 x in, q8_K out), then the GEMV."""
    return sum(gemv_bytes(n, k) + quant_bytes(k) for _, _, n, k, _ in mats)


def fused_step_bytes(mats):
    """The headline step, one fused launch: weights and f32 x read once, y
    written once (the q8_K codes never leave the chip)."""
    return sum(n * (k // QK) * Q4K_BYTES + 4 * k + 4 * n for _, _, n, k, _ in mats)


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
                 "--format=csv,noheader,nounits", "-lms", "100"],
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

def host_inputs():
    import gen
    mats, total = mat_list()
    host_w = np.empty(total, dtype=np.uint8)
    for idx, (layer, j, n, k, off) in enumerate(mats):
        sz = n * (k // QK) * Q4K_BYTES
        gen.q4K_blocks(SEED, idx, n, k, out=host_w[off:off + sz].reshape(n, -1))
    xs = [gen.normal_f32(SEED, 1000 + idx, 1, k) for idx, (_, _, _, k, _) in enumerate(mats)]
    return mats, host_w, xs


# --------------------------------------------------------------- oracle

def cpu_oracle_pass(mats, host_w, xs, count, threads):
    import oracle
    oracle.set_threads(threads)
    for idx in range(count):
        _, _, n, k, off = mats[idx]
        sz = n * (k // QK) * Q4K_BYTES
        xq = oracle.quantize_q8K(xs[idx])
        oracle.gemm_q4K_f32(host_w[off:off + sz], xq, 1, n, k)


def oracle_rate(mats, host_w, xs, budget_s, threads=None):
    """Times the oracle (as it stands) on the first matrices of the set,
    as many full passes as fit the budget; returns (GB/s, sample text, cores)."""
    cores = len(os.sched_getaffinity(0))
    th = cores if threads is None else threads
    t0 = time.perf_counter()
    cpu_oracle_pass(mats, host_w, xs, 7, th)              # one layer, warm
    per_layer = time.perf_counter() - t0
    count = 7 * max(1, min(N_LAYERS, int(budget_s / 4 / max(per_layer, 1e-6))))
    reps, t0 = 0, time.perf_counter()
    while True:
        cpu_oracle_pass(mats, host_w, xs, count, th)
        reps += 1
        el = time.perf_counter() - t0
        if el > budget_s / 2:
            break
    alg = step_bytes(mats[:count]) * reps
    sample = ("%d of 196 matrices (%d of 28 layers) x %d passes: q8_K quantize + q4_K f32 oracle "
              "GEMV, %s, %.1f s" % (count, count // 7, reps,
                                    "one thread" if th == 1 else "OpenMP over output rows, %d threads" % th, el))
    return alg / el / 1e9, sample, cores


def oracle_details(cores):
    """The oracle timed the ways the pages time the CPU path: the q8_K
    quantizer alone on the 512x1024 prefill shape, single-threaded and on all
    cores, and the q6_K output heads (151936 x 2048 and x 4096) on 1024-row
    slices at m = 1, 8 and 512, reported per multiply-add and extrapolated to
    the whole head."""
    import gen
    import oracle
    out = {}
    x = gen.normal_f32(2, 0, 512, 1024)
    for label, th in (("single_thread", 1), ("openmp", cores)):
        oracle.set_threads(th)
        oracle.quantize_q8K(x)
        reps, t0 = 0, time.perf_counter()
        while reps < 3 or time.perf_counter() - t0 < 0.5:
            oracle.quantize_q8K(x)
            reps += 1
        out["quantize_512x1024_" + label] = {"us": (time.perf_counter() - t0) / reps * 1e6, "threads": th}
    heads = []
    oracle.set_threads(cores)
    for seed, k in ((3, 2048), (4, 4096)):
        w = gen.q6K_blocks(seed, 0, 1024, k)
        for m in (1, 8, 512):
            xq = oracle.quantize_q8K(gen.normal_f32(seed, 50 + m, m, k))
            reps, t0 = 0, time.perf_counter()
            while reps < 1 or time.perf_counter() - t0 < 0.3:
                oracle.gemm_q6K_f32(w, xq, m, 1024, k)
                reps += 1
            el = (time.perf_counter() - t0) / reps
            heads.append({"shape": "q6_K 1024 of 151936 rows x %d" % k, "m": m, "s_per_slice": el,
                          "mac_per_s": 1024.0 * k * m / el,
                          "full_head_s_extrapolated": el * 151936 / 1024, "threads": cores})
    out["q6K_head_slices"] = heads
    return out


def run_reference(args, rank):
    if rank != 0:
        return
    import oracle
    mats, host_w, xs = host_inputs()
    cores = len(os.sched_getaffinity(0))
    t0 = time.perf_counter()
    cpu_oracle_pass(mats, host_w, xs, 7, cores)
    per_layer = time.perf_counter() - t0
    # a step is a bounded sample so that warm-up + steps end within minutes
    count = 7 * max(1, min(N_LAYERS, int(1.0 / max(per_layer, 1e-6))))
    for _ in range(args.warmup):
        cpu_oracle_pass(mats, host_w, xs, count, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_oracle_pass(mats, host_w, xs, count, cores)
    el = time.perf_counter() - t0
    val = step_bytes(mats[:count]) * args.steps / el / 1e9
    sample = ("%d of 196 matrices per step: q8_K quantize + q4_K f32 oracle GEMV, "
              "OpenMP over output rows" % count)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "s8 x u4 -> s32 -> f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "m": 1, "seed": SEED},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "threads": oracle.max_threads(), "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# --------------------------------------------------------------- one case

def time_case(args):
    """Times one entry point on one shape: weights rotated through enough
    copies to exceed three times the L2, CUDA events on the launch stream."""
    import torch
    import gen
    import quant_packed_gemv_gb300 as q
    kind, fmt, n, k = args.case[0], args.case[1], int(args.case[2]), int(args.case[3])
    torch.cuda.set_device(0)
    nb = k // QK
    bpb = FMT_BYTES[fmt]
    wbytes = n * nb * bpb
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    copies = max(1, -(-3 * l2 // wbytes))
    w_host = getattr(gen, "%s_blocks" % fmt)(4, 0, n, k)
    ws = [torch.from_numpy(w_host).cuda() for _ in range(copies)]
    if kind == "gemv_x16":
        # the row-interleaved layout: repack every copy once (not timed)
        packed = []
        for wd in ws:
            wx = torch.empty(getattr(q, "plm_%s_x16_size" % fmt)(n, k), dtype=torch.uint8, device="cuda")
            getattr(q, "plm_%s_to_x16" % fmt)(wd, wx, n, k)
            packed.append(wx)
        torch.cuda.synchronize()
        ws = packed
    if kind == "gemv_x16":
        fn = getattr(q, "plm_gemv_%s_x16" % fmt)
    elif kind == "gemm_ws":
        # the workspace form with the split-K workspace size
        fws = getattr(q, "plm_gemm_%s_ws" % fmt)
        works = {}

        def fn(w, xq, y, m, n, k, stream):
            if m not in works:
                need = q.plm_gemm_workspace_size_split(fmt, m, n, k)
                works[m] = (torch.empty(max(need, 256), dtype=torch.uint8, device="cuda"), need)
            wk, need = works[m]
            fws(w, xq, y, m, n, k, wk if need else None, need, stream=stream)
    else:
        fn = getattr(q, "plm_%s_%s" % (kind, fmt))
    q.plm_set_overlap(args.overlap)
    stream = torch.cuda.Stream()
    for m in args.m:
        x = torch.from_numpy(gen.normal_f32(4, 9, m, k)).cuda()
        xq = torch.empty(m * nb * Q8K_BYTES, dtype=torch.uint8, device="cuda")
        y = torch.empty(m * n, dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            q.plm_quantize_q8K(x, xq, m, k, stream=stream)
            for i in range(max(args.warmup, 3)):
                fn(ws[i % copies], xq, y, m, n, k, stream=stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(args.steps):
                    fn(ws[i % copies], xq, y, m, n, k, stream=stream)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / args.steps
        byt = wbytes + m * nb * Q8K_BYTES + m * n * 4
        print(json.dumps({"case": "%s_%s" % (kind, fmt), "n": n, "k": k, "m": m, "us": us,
                          "gbs": byt / us / 1e3, "tops": 2.0 * m * n * k / us / 1e6,
                          "copies": copies, "fault": q.plm_device_fault()}), flush=True)


def recorded_counters(key):
    """The committed ncu record of one kernel (DRAM bytes per launch and other
    counters), or None when the kernel sources changed since the capture."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))[key]
        h = hashlib.sha256()
        for p in rec["sources"]:
            h.update(open(os.path.join(ROOT, p), "rb").read())
        return rec if h.hexdigest()[:16] == rec["sources_sha256_16"] else None
    except (OSError, ValueError, KeyError):
        return None


def recorded_traffic(key):
    """DRAM bytes per launch from the committed ncu record, or None when the
    kernel sources changed since the capture."""
    rec = recorded_counters(key)
    return rec["dram_bytes_per_launch"] if rec else None


# --------------------------------------------------------------- other configs

class ShapeTimer:
    """Times single entry points on one shape with the weights rotated
    through enough copies to exceed three times the L2; CUDA events on the
    launch stream.  GEMMs use the caller-workspace form with a workspace
    allocated once (allocation is not part of the timed work)."""

    def __init__(self, torch, q, peaks):
        self.torch, self.q, self.peaks = torch, q, peaks
        self.l2 = torch.cuda.get_device_properties(0).L2_cache_size
        self.stream = torch.cuda.Stream()

    def weights(self, fmt, seed, n, k):
        import gen
        host = getattr(gen, "%s_blocks" % fmt)(seed, 0, n, k)
        copies = max(1, -(-3 * self.l2 // host.nbytes))
        return [self.torch.from_numpy(host).cuda() for _ in range(copies)], host.nbytes

    def x16(self, fmt, ws_list, n, k):
        """The same weight copies repacked into the row-interleaved x16 layout."""
        torch, q = self.torch, self.q
        out = []
        for w in ws_list:
            wx = torch.empty(getattr(q, "plm_%s_x16_size" % fmt)(n, k), dtype=torch.uint8, device="cuda")
            getattr(q, "plm_%s_to_x16" % fmt)(w, wx, n, k)
            out.append(wx)
        torch.cuda.synchronize()
        return out

    def run(self, fmt, ws_list, wbytes, n, k, m, steps, warmup, layout="ggml"):
        import gen
        torch, q = self.torch, self.q
        nb = k // QK
        x = torch.from_numpy(gen.normal_f32(7, m, m, k)).cuda()
        xq = torch.empty(m * nb * Q8K_BYTES, dtype=torch.uint8, device="cuda")
        y = torch.empty(m * n, dtype=torch.float32, device="cuda")
        gemv = m <= 8
        # GEMM: the workspace form (pre-pass, K split where it pays) or, with
        # layout "plain", the entry without a workspace (codes widened in the kernel)
        plain = gemv or layout == "plain"
        need = 0 if plain else q.plm_gemm_workspace_size_split(fmt, m, n, k)
        work = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        fn = getattr(q, ("plm_gemv_%s" if gemv else "plm_gemm_%s" if plain else "plm_gemm_%s_ws") % fmt)
        if layout == "x16":
            fn = getattr(q, "plm_gemv_%s_x16" % fmt)
        s = self.stream

        def call(i):
            w = ws_list[i % len(ws_list)]
            if plain:
                fn(w, xq, y, m, n, k, stream=s)
            else:
                fn(w, xq, y, m, n, k, work, need, stream=s)
        with torch.cuda.stream(s):
            q.plm_quantize_q8K(x, xq, m, k, stream=s)
            for i in range(warmup):
                call(i)
            torch.cuda.synchronize()
            # the timed calls replay from a CUDA graph, so host-side launch cost
            # does not gap the device timeline
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(steps):
                    call(i)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / steps
        byt = wbytes + m * nb * Q8K_BYTES + m * n * 4
        r = {"fmt": fmt, "n": n, "k": k, "m": m, "us": round(us, 3),
             "entry": fn.__name__}
        if gemv:
            gbs = byt / us / 1e3
            r.update({"GB_per_s": round(gbs, 1), "frac_hbm": round(gbs / self.peaks["hbm_gbs"], 4),
                      "weights_per_s": n * k / (us * 1e-6)})
        else:
            tops = 2.0 * m * n * k / us / 1e6
            r.update({"TOPS": round(tops, 1),
                      "frac_f16_dense": round(tops / self.peaks["bf16_tflops"], 4)})
        return r


def time_pair(T, wg_list, wu_list, n, k, m, steps, warmup, plain=False):
    """The prefill gate/up pair with SwiGLU on one shape (plm_gemm_q4K_swiglu_ws,
    or with plain=True plm_gemm_q4K_swiglu: no workspace, the combine in the up
    GEMM's epilogue), weights rotated as for ShapeTimer, a CUDA graph of
    `steps` calls."""
    import gen
    torch, q = T.torch, T.q
    nb = k // QK
    x = torch.from_numpy(gen.normal_f32(8, m, m, k)).cuda()
    xq = torch.empty(m * nb * Q8K_BYTES, dtype=torch.uint8, device="cuda")
    h = torch.empty(m * n, dtype=torch.float32, device="cuda")
    need = 0 if plain else q.plm_gemm_swiglu_workspace_size(m, n, k)
    work = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    s = T.stream

    def call(i):
        if plain:
            q.plm_gemm_q4K_swiglu(wg_list[i % len(wg_list)], wu_list[i % len(wu_list)], xq, h, m, n, k, stream=s)
        else:
            q.plm_gemm_q4K_swiglu_ws(wg_list[i % len(wg_list)], wu_list[i % len(wu_list)], xq, h, m, n, k,
                                     work if need else None, need, stream=s)
    with torch.cuda.stream(s):
        q.plm_quantize_q8K(x, xq, m, k, stream=s)
        for i in range(warmup):
            call(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(steps):
                call(i)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        g.replay()
        e1.record(s)
        torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / steps
    tops = 4.0 * m * n * k / us / 1e6   # two matrices
    return {"fmt": "q4K", "n": n, "k": k, "m": m, "us": round(us, 3),
            "entry": "plm_gemm_q4K_swiglu" if plain else "plm_gemm_q4K_swiglu_ws",
            "TOPS": round(tops, 1), "frac_f16_dense": round(tops / T.peaks["bf16_tflops"], 4)}


def run_extras(torch, q, peaks):
    """Prefill GEMMs (Qwen3 m=512 shapes), the q6_K output head at m = 1, 8,
    512, and the Qwen3-8B sweep over m, each shape timed alone."""
    T = ShapeTimer(torch, q, peaks)
    out = {}
    res = []
    for n, k in [(1024, 1024), (6144, 2048), (2048, 6144)]:
        ws, wb = T.weights("q4K", 2, n, k)
        res.append(T.run("q4K", ws, wb, n, k, 512, 10, 3))
        del ws
    out["prefill_gemm_q4K_m512"] = res
    ws, wb = T.weights("q6K", 3, 151936, 2048)
    out["q6K_head_151936x2048"] = [T.run("q6K", ws, wb, 151936, 2048, m, 10 if m <= 8 else 4, 2)
                                   for m in (1, 8, 512)]
    wx = T.x16("q6K", ws, 151936, 2048)
    out["q6K_head_151936x2048"] += [T.run("q6K", wx, wb, 151936, 2048, m, 10, 2, layout="x16") for m in (1, 8)]
    del ws, wx
    sweep = []
    for fmt, n, k in [("q4K", 12288, 4096), ("q4K", 4096, 12288), ("q6K", 151936, 4096)]:
        ws, wb = T.weights(fmt, 4, n, k)
        for m in (1, 2, 4, 8, 64, 512, 2048):
            steps = 10 if m <= 8 else (5 if n * k * m < 3e11 else 2)
            sweep.append(T.run(fmt, ws, wb, n, k, m, steps, 1 if m > 512 else 2))
        # the GEMM entry without a workspace (activation codes widened in the kernel, no K split)
        for m in (64, 512, 2048):
            steps = 5 if n * k * m < 3e11 else 2
            sweep.append(T.run(fmt, ws, wb, n, k, m, steps, 1 if m > 512 else 2, layout="plain"))
        # the decode GEMV on the row-interleaved layout (tensor-core tile)
        wx = T.x16(fmt, ws, n, k)
        for m in (1, 2, 4, 8):
            sweep.append(T.run(fmt, wx, wb, n, k, m, 10, 2, layout="x16"))
        del ws, wx
        torch.cuda.empty_cache()
    out["sweep_qwen3_8b"] = sweep
    # the q5_K rung on the Qwen3-8B gate/up shape: decode GEMV and prefill GEMM
    ws, wb = T.weights("q5K", 5, 12288, 4096)
    out["q5K_12288x4096"] = [T.run("q5K", ws, wb, 12288, 4096, m, 10 if m <= 8 else 3, 2) for m in (1, 8, 512)]
    del ws
    # the prefill gate/up pair with the SwiGLU epilogue (workspace form: two GEMMs and one
    # elementwise pass; plain form: the combine in the up GEMM's epilogue)
    wg, _ = T.weights("q4K", 6, 12288, 4096)
    wu, _ = T.weights("q4K", 7, 12288, 4096)
    out["prefill_swiglu_q4K_12288x4096"] = [time_pair(T, wg, wu, 12288, 4096, m, 5 if m < 2048 else 3, 2, plain)
                                            for plain in (False, True) for m in (64, 512, 2048)]
    del wg, wu
    torch.cuda.empty_cache()
    # the q2_K and q3_K rungs: decode GEMV, and the tensor-core GEMM (workspace and plain forms)
    for fmt in ("q3K", "q2K"):
        ws, wb = T.weights(fmt, 5, 12288, 4096)
        out["%s_12288x4096" % fmt] = ([T.run(fmt, ws, wb, 12288, 4096, m, 10, 2) for m in (1, 8)] +
                                      [T.run(fmt, ws, wb, 12288, 4096, m, 3, 2, layout=lay)
                                       for lay in ("ggml", "plain") for m in (512, 2048)])
        del ws
    return out


def gemm_roofline(configs, peaks, peak_src):
    """Roofline of the dominant prefill kernel: the q4_K tensor-core GEMM on
    the Qwen3-8B gate/up shape 12288 x 4096 at m = 2048 in its workspace
    form, from the sweep's CUDA-event time per call (the call is the
    activation pre-pass, about 2 %, then the GEMM kernel as its main grid and
    the short last wave's launch, so the kernel's own rate is slightly
    higher); traffic and tensor-pipe activity per call from the ncu record."""
    row = next((r for r in configs.get("sweep_qwen3_8b", [])
                if r["fmt"] == "q4K" and r["n"] == 12288 and r["k"] == 4096 and r["m"] == 2048
                and r["entry"] == "plm_gemm_q4K_ws"), None)
    if row is None:
        return None
    peak = peaks["bf16_tflops"]
    flops = 2.0 * row["m"] * row["n"] * row["k"]
    achieved = flops / (row["us"] * 1e-6) / 1e12
    rec = recorded_counters("gemm_q4K_12288x4096_m2048")
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": rec.get("dram_bytes_per_launch") if rec else None,
            "tensor_pipe_active_pct": rec.get("tensor_pipe_active_pct") if rec else None,
            "peak_source": "measured bf16 dense (burst); f16, the kind the kernel runs, has the same nominal rate"
                           if peak_src == "measured" else "fallback",
            "kernel": "gemm_tm_kernel<q4_K> (tcgen05.mma kind::f16 on exact integer-valued operands, A in tensor memory)",
            "shape": "q4_K 12288x4096, m=2048", "flops_per_call": flops, "avg_call_us": row["us"]}


# --------------------------------------------------------------- main arm

class Step:
    """Device buffers of one step and the C-ABI call sequences over them."""

    def __init__(self, torch, dev, mats, host_w, xs):
        self.mats = mats
        self.w = [torch.from_numpy(host_w).to(dev) for _ in range(2)]
        self.xoff, self.qoff, self.yoff = [], [], []
        xo = qo = yo = 0
        for (_, _, n, k, _) in mats:
            self.xoff.append(xo)
            self.qoff.append(qo)
            self.yoff.append(yo)
            xo += k
            qo += k // QK * Q8K_BYTES
            yo += n
        self.x_host = torch.from_numpy(np.concatenate([x.ravel() for x in xs])).pin_memory()
        self.x = self.x_host.to(dev)
        self.xq = torch.empty(qo, dtype=torch.uint8, device=dev)
        self.y = torch.empty(yo, dtype=torch.float32, device=dev)
        self.y_host = torch.empty(yo, dtype=torch.float32).pin_memory()
        self.nchunks = xo // QK
        self.fused = None
        self.sets = None
        # grouped problem lists, one per weight copy
        self.problems = []
        for c in range(2):
            wp = self.w[c].data_ptr()
            self.problems.append([(wp + off, self.xq.data_ptr() + self.qoff[i],
                                   self.y.data_ptr() + 4 * self.yoff[i], n, k)
                                  for i, (_, _, n, k, off) in enumerate(mats)])

    def add_io_sets(self, torch, dev):
        """Two activation/output sets (the first is x, xq, y) for the end-to-end
        loop, whose host copies of one step overlap the other step's compute."""
        xq2 = torch.empty_like(self.xq)
        x_host2 = self.x_host.clone().pin_memory()
        self.sets = [dict(x=self.x, xq=self.xq, y=self.y, x_host=self.x_host, y_host=self.y_host),
                     dict(x=x_host2.to(dev), xq=xq2, y=torch.empty_like(self.y), x_host=x_host2,
                          y_host=torch.empty_like(self.y_host).pin_memory())]
        for st in self.sets:
            st["fused"] = [[(self.w[c].data_ptr() + off, st["x"].data_ptr() + 4 * self.xoff[i],
                             st["y"].data_ptr() + 4 * self.yoff[i], n, k)
                            for i, (_, _, n, k, off) in enumerate(self.mats)] for c in range(2)]

    def run_set(self, q, b, copy, stream):
        """The headline step on activation/output set b: one fused launch."""
        q.plm_quantize_gemv_q4K_grouped(self.sets[b]["fused"][copy], 1, stream=stream)

    def run_chain_fused(self, q, copy, stream):
        """Decode order with the fused producer: one launch per dependent stage."""
        wp = self.w[copy].data_ptr()
        for layer in range(N_LAYERS):
            for first, cnt in CHAIN:
                i = layer * 7 + first
                _, _, _, k, off = self.mats[i]
                n = sum(self.mats[i + j][2] for j in range(cnt))
                q.plm_quantize_gemv_q4K(wp + off, self.x.data_ptr() + 4 * self.xoff[i],
                                        self.y.data_ptr() + 4 * self.yoff[i], 1, n, k, stream=stream)

    def fused_problems(self, copy):
        wp, xp, yp = self.w[copy].data_ptr(), self.x.data_ptr(), self.y.data_ptr()
        return [(wp + off, xp + 4 * self.xoff[i], yp + 4 * self.yoff[i], n, k)
                for i, (_, _, n, k, off) in enumerate(self.mats)]

    def gate_up(self, copy):
        """The 28 ffn gate/up pairs (3072x1024 each) on the gate's activations:
        as SwiGLU pairs, and as the same 56 matrices for plain grouped GEMVs."""
        wp, qp, yp = self.w[copy].data_ptr(), self.xq.data_ptr(), self.y.data_ptr()
        pairs, plain = [], []
        for layer in range(N_LAYERS):
            ig, iu = layer * 7 + 4, layer * 7 + 5
            _, _, n, k, og = self.mats[ig]
            ou = self.mats[iu][4]
            xq = qp + self.qoff[ig]
            pairs.append((wp + og, wp + ou, xq, yp + 4 * self.yoff[ig], n, k))
            plain.append((wp + og, xq, yp + 4 * self.yoff[ig], n, k))
            plain.append((wp + ou, xq, yp + 4 * self.yoff[iu], n, k))
        return pairs, plain

    def run_fused(self, q, copy, stream):
        """One launch: each CTA quantizes its activations and runs the GEMV."""
        q.plm_quantize_gemv_q4K_grouped(self.fused[copy], 1, stream=stream)

    def run(self, q, copy, stream, quantize=True, gemv=True):
        if quantize:
            q.plm_quantize_q8K(self.x, self.xq, self.nchunks, QK, stream=stream)
        if gemv:
            q.plm_gemv_q4K_grouped(self.problems[copy], 1, stream=stream)

    def run_chain(self, q, copy, stream):
        """Decode order: per layer, quantize + GEMV for each dependent stage."""
        wp = self.w[copy].data_ptr()
        for layer in range(N_LAYERS):
            for first, cnt in CHAIN:
                i = layer * 7 + first
                _, _, _, k, off = self.mats[i]
                n = sum(self.mats[i + j][2] for j in range(cnt))
                xq = self.xq.data_ptr() + self.qoff[i]
                q.plm_quantize_q8K(self.x.data_ptr() + 4 * self.xoff[i], xq, 1, k, stream=stream)
                q.plm_gemv_q4K(wp + off, xq, self.y.data_ptr() + 4 * self.yoff[i], 1, n, k, stream=stream)


def main():
    args = parse()
    if args.case:
        time_case(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    import torch
    import quant_packed_gemv_gb300 as q
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    pg = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        pg = dist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q.load()

    mats, host_w, xs = host_inputs()
    st = Step(torch, dev, mats, host_w, xs)
    stream = torch.cuda.Stream(device=dev)

    q.plm_set_overlap(args.overlap)
    st.fused = [st.fused_problems(c) for c in range(2)]
    gate_up = [st.gate_up(c) for c in range(2)]
    K = args.steps
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            if not args.no_two_launch:
                st.run(q, i % 2, stream)
            st.run_fused(q, i % 2, stream)
            q.plm_gemv_q4K_swiglu_grouped(gate_up[i % 2][0], 1, stream=stream)
            q.plm_gemv_q4K_grouped(gate_up[i % 2][1], 1, stream=stream)
            if not args.no_chain:
                st.run_chain(q, i % 2, stream)
    torch.cuda.synchronize()

    def capture(fn, steps):
        """One CUDA graph of `steps` consecutive steps, weight copies alternating."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(steps):
                fn(s)
        return g

    run_step = lambda s: st.run(q, s % 2, stream)
    run_gemv = lambda s: st.run(q, s % 2, stream, quantize=False)
    run_fused = lambda s: st.run_fused(q, s % 2, stream)
    run_swiglu = lambda s: q.plm_gemv_q4K_swiglu_grouped(gate_up[s % 2][0], 1, stream=stream)
    run_gateup = lambda s: q.plm_gemv_q4K_grouped(gate_up[s % 2][1], 1, stream=stream)
    run_chain = lambda s: st.run_chain(q, s % 2, stream)
    # the timed graphs: K steps each; single-step graphs: the end-to-end loop
    # and a per-step comparison
    fused_g = capture(run_fused, K)
    step_g = None if args.no_two_launch else capture(run_step, K)
    gemv_g = None if args.no_two_launch else capture(run_gemv, K)
    swiglu_g, gateup_g = capture(run_swiglu, K), capture(run_gateup, K)
    chain_g = None if args.no_chain else capture(run_chain, K)
    chain_fused_g = None if args.no_chain else capture(lambda s: st.run_chain_fused(q, s % 2, stream), K)
    single = [capture(lambda s, c=c: st.run_fused(q, c, stream), 1) for c in range(2)]
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

    def timed_graph(g):
        g.replay()                       # untimed: graph upload
        torch.cuda.synchronize()
        return timed(lambda s: g.replay(), 1)

    h2d = st.x_host.numel() * 4
    d2h = st.y_host.numel() * 4

    def e2e_step(s):
        st.x.copy_(st.x_host, non_blocking=True)
        single[s % 2].replay()
        st.y_host.copy_(st.y, non_blocking=True)

    # End to end, pipelined: every step copies its activations in from pinned
    # host memory and its outputs out, on a copy stream, with two
    # activation/output sets so that step s+1's input copy and step s's output
    # copy overlap the compute; the K steps are captured as one graph.
    st.add_io_sets(torch, dev)
    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_pipelined(steps):
        sets = st.sets

        def h2d_copy(s):
            with torch.cuda.stream(copy_stream):
                sets[s % 2]["x"].copy_(sets[s % 2]["x_host"], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(copy_stream)
            return ev
        fork = torch.cuda.Event()
        fork.record(stream)
        copy_stream.wait_event(fork)
        ev_in = h2d_copy(0)
        for s in range(steps):
            b = s % 2
            nxt = h2d_copy(s + 1) if s + 1 < steps else None   # after the output copy of step s - 1
            stream.wait_event(ev_in)
            st.run_set(q, b, s % 2, stream)
            done = torch.cuda.Event()
            done.record(stream)
            copy_stream.wait_event(done)
            with torch.cuda.stream(copy_stream):
                sets[b]["y_host"].copy_(sets[b]["y"], non_blocking=True)
            ev_in = nxt
        join = torch.cuda.Event()
        join.record(copy_stream)
        stream.wait_event(join)

    with torch.cuda.stream(stream):
        e2e_pipelined(2)
    torch.cuda.synchronize()
    e2e_g = capture(lambda s: e2e_pipelined(K) if s == 0 else None, 1)
    # End to end without copy calls: the fused step reads the activations from
    # pinned host memory and writes y to pinned host memory itself (the GPU
    # reaches host memory coherently over the CPU-GPU link); the same bytes
    # cross the link inside the timed region
    zc = [[(st.w[c].data_ptr() + off, st.x_host.data_ptr() + 4 * st.xoff[i], st.y_host.data_ptr() + 4 * st.yoff[i],
            n, kk) for i, (_, _, n, kk, off) in enumerate(mats)] for c in range(2)]
    with torch.cuda.stream(stream):
        for i in range(3):
            q.plm_quantize_gemv_q4K_grouped(zc[i % 2], 1, stream=stream)
    torch.cuda.synchronize()
    zc_g = capture(lambda s: q.plm_quantize_gemv_q4K_grouped(zc[s % 2], 1, stream=stream), K)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            single[s % 2].replay()
            e2e_step(s)
        torch.cuda.synchronize()
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        ms = timed_graph(step_g) if step_g is not None else None
        gemv_ms = timed_graph(gemv_g) if gemv_g is not None else None
        fused_ms = timed_graph(fused_g)
        swiglu_ms = timed_graph(swiglu_g)
        gateup_ms = timed_graph(gateup_g)
        chain_ms = timed_graph(chain_g) if chain_g is not None else None
        chain_fused_ms = timed_graph(chain_fused_g) if chain_fused_g is not None else None
        e2e_pipe_ms = timed_graph(e2e_g)
        zc_ms = timed_graph(zc_g)
        single_ms = timed(lambda s: single[s % 2].replay(), K)
        t0 = time.perf_counter()
        e2e_ms = timed(e2e_step, K)
        e2e_wall = (time.perf_counter() - t0) * 1e3
        clocks = sampler.stop()
    fault = q.plm_device_fault()

    # the headline step: the fused producer + GEMV, one grouped launch per 256 problems
    alg = fused_step_bytes(mats)
    two_alg = step_bytes(mats)
    gemv_alg = sum(gemv_bytes(n, k) for _, _, n, k, _ in mats)
    ms_step = fused_ms / args.steps
    value = world * alg / (ms_step * 1e-3) / 1e9
    launches_grouped = -(-len(mats) // 256)                  # grouped launches per step
    fused_launch_ms = ms_step / launches_grouped
    achieved = alg / launches_grouped / (fused_launch_ms * 1e-3) / 1e9
    gemv_launch_ms = gemv_ms / args.steps / launches_grouped if gemv_ms is not None else None
    gemv_achieved = gemv_alg / launches_grouped / (gemv_launch_ms * 1e-3) / 1e9 if gemv_ms is not None else None
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    e2e_ms_step = max(e2e_ms, e2e_wall) / args.steps
    chain_step = chain_ms / args.steps if chain_ms is not None else None
    swiglu_bytes = sum(2 * n * (k // QK) * Q4K_BYTES + (k // QK) * Q8K_BYTES + 4 * n
                       for (_, j, n, k, _) in mats if j == 4)
    chain_fused_bytes = sum(sum(mats[l * 7 + f + j][2] for j in range(c)) * (mats[l * 7 + f][3] // QK) * Q4K_BYTES
                            + 4 * mats[l * 7 + f][3] + 4 * sum(mats[l * 7 + f + j][2] for j in range(c))
                            for l in range(N_LAYERS) for f, c in CHAIN)
    chain_bytes = sum(gemv_bytes(sum(mats[l * 7 + f + j][2] for j in range(c)), mats[l * 7 + f][3])
                      + quant_bytes(mats[l * 7 + f][3]) for l in range(N_LAYERS) for f, c in CHAIN)

    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "s8 x u4 -> s32 -> f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "m": 1, "seed": SEED,
                   "weights_mb": sum(n * (k // QK) * Q4K_BYTES for _, _, n, k, _ in mats) / 1e6,
                   "l2": "inputs larger than L2: two 247.7 MB weight copies, alternate steps",
                   "launch": "per step %d launch(es) of plm_quantize_gemv_q4K_grouped (each CTA quantizes "
                             "its f32 activations to q8_K, then runs the GEMV); the K timed steps replay as "
                             "one CUDA graph" % launches_grouped,
                   "overlap": {0: "plain stream order", 1: "early launch",
                               2: "early launch with weight prefetch"}[args.overlap]},
        "ms_per_step_one_graph_per_step": single_ms / args.steps,
        "weights_per_s": world * sum(n * k for _, _, n, k, _ in mats) / (ms_step * 1e-3),
        "gpu_launches": launches_grouped * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic("gemv_q4K_fused_grouped_m1"),
                     "peak_source": peak_src,
                     "kernel": "q4lane::lane_kernel<m=1, 16 warps, grouped, f32 activations quantized in the CTA> "
                               "(q4_K, one lane per block)",
                     "avg_launch_us": fused_launch_ms * 1e3,
                     "bytes_per_launch": alg / launches_grouped},
        "decode_set_two_launch": None if ms is None else {
            "value": world * two_alg / (ms / args.steps * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": ms / args.steps, "launches_per_step": 1 + launches_grouped,
            "bytes_per_step": two_alg,
            "what": "the same step as plm_quantize_q8K then plm_gemv_q4K_grouped (q8_K through HBM)",
            "gemv_roofline": {"bound": "hbm", "achieved": gemv_achieved, "peak": peak, "unit": "GB/s",
                              "frac": gemv_achieved / peak, "traffic": recorded_traffic("gemv_q4K_grouped_m1"),
                              "kernel": "q4lane::lane_kernel<m=1, 16 warps, grouped> on q8_K activations",
                              "avg_launch_us": gemv_launch_ms * 1e3,
                              "bytes_per_launch": gemv_alg / launches_grouped}},
        "decode_chain": None if chain_step is None else {
            "value": world * chain_bytes / (chain_step * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": chain_step, "launches_per_step": 8 * N_LAYERS,
            "what": "28 layers x 4 dependent (quantize, GEMV) stages, CUDA graph"},
        "decode_chain_fused": None if chain_fused_ms is None else {
            "value": world * chain_fused_bytes / (chain_fused_ms / args.steps * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": chain_fused_ms / args.steps, "launches_per_step": 4 * N_LAYERS,
            "what": "the same chain with plm_quantize_gemv_q4K: one launch per dependent stage"},
        "swiglu_gate_up": {
            "value": world * swiglu_bytes / (swiglu_ms / args.steps * 1e-3) / 1e9, "unit": "GB/s",
            "us_per_launch": swiglu_ms / args.steps * 1e3,
            "two_matrix_grouped_gemv_us": gateup_ms / args.steps * 1e3,
            "what": "28 q4_K gate/up pairs (3072x1024), m=1: plm_gemv_q4K_swiglu_grouped writes "
                    "h = silu(g)*u; compared with one grouped GEMV over the same 56 matrices"},
        "e2e": {"value": world * alg / (e2e_pipe_ms / args.steps * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_pipe_ms / args.steps,
                "how": "per step: x copied in from pinned host memory, the fused quantize + grouped GEMV, "
                       "y copied out; copies on a second stream with two buffer sets so they overlap the "
                       "compute; the K steps captured as one CUDA graph",
                "zero_copy": {"value": world * alg / (zc_ms / args.steps * 1e-3) / 1e9,
                              "ms_per_step": zc_ms / args.steps,
                              "how": "the fused step reading x from and writing y to pinned host memory "
                                     "directly, no copy calls; same bytes per step"},
                "serial": {"value": world * alg / (e2e_ms_step * 1e-3) / 1e9, "ms_per_step": e2e_ms_step,
                           "how": "copy in, one-step graph, copy out, on one stream, no overlap"}},
        "clocks": clocks,
        "device_fault": fault,
    }
    s8_tops, f16_tflops = q.plm_probe_mma_rates()
    tc_cyc, tc_cyc_wait, tc_tflops = q.plm_probe_tcgen05_rate()
    out["peaks"] = {"hbm_gbs": peak, "hbm_source": peak_src,
                    "bf16_tflops": peaks.get("bf16_tflops", 1900.0),
                    "int8_mma_tops": s8_tops, "f16_mma_sync_tflops": f16_tflops,
                    "tcgen05_f16_128x128x16": {"cycles_per_mma": tc_cyc, "cycles_per_mma_wait_after_commit": tc_cyc_wait,
                                               "tflops_zero_operands": tc_tflops},
                    "note": "context only: legacy mma.sync rates and the GEMM's tcgen05 MMA (one thread, commit "
                            "every four; zero operands) measured live (tcgen05 has no int8 kind on sm_103a); the "
                            "GEMM's roofline is the measured bf16 dense peak (f16 has the same nominal rate)"}
    if rank == 0 and not args.no_extras:
        del st
        torch.cuda.empty_cache()
        out["configs"] = run_extras(torch, q, out["peaks"])
        out["roofline_gemm"] = gemm_roofline(out["configs"], out["peaks"], peak_src)
    if rank == 0 and not args.no_cpu_baseline:
        val, sample, cores = oracle_rate(mats, host_w, xs, 12.0)
        import oracle
        out["cpu_baseline"] = {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                               "threads": oracle.max_threads(), "sample": sample}
        val1, sample1, _ = oracle_rate(mats, host_w, xs, 6.0, threads=1)
        out["cpu_baseline"]["single_thread"] = {"value": val1, "unit": "GB/s", "threads": 1, "sample": sample1}
        out["cpu_baseline"].update(oracle_details(cores))
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
