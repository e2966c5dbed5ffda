"""Throughput of the Swin shifted-window attention block on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one forward of the whole block (cyclic shift, partition, QKV
projection, windowed attention with relative bias and shift mask, softmax,
P.V, reverse, roll back, output projection) over one batch of synthetic
inputs already resident in HBM.  Default workload: the Swin-T stage-1 shifted
block (B=64, 56x56 tokens, C=96, 3 heads, M=7, s=3, bf16, V1).  Inputs are
rotated over several buffer sets whose total exceeds twice the L2, so no step
reads what the previous one left in L2.  Multi-GPU: one process per GPU
(torchrun), each rank runs its own batch (weak scaling, no collective in the
data path), times are the max over ranks.

Prints one JSON line: tokens/s (value), TFLOP/s, the roofline of the dominant
kernel (CUDA events inside this run), the whole block's roofline fraction, the
end-to-end number through swin_wattn_forward_host (pinned host buffers, copies
inside the timed region), the clocks seen during the run, and the float64
oracle timed on the host cores on a bounded sample (cpu_baseline).
--impl reference times that oracle alone as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from vision_transformer_shifted_gb300.inputs import V1, V2, WORKLOADS, generate  # noqa: E402

L2_BYTES = 129 * 1024 * 1024

# DRAM bytes (read + write) per launch from ncu captures, keyed by
# workload and kernel, with the sha1 prefix of the kernel source they were taken
# on: reported only while the source is unchanged.
PROFILED_TRAFFIC = {
    ("swin_t_s1", "fused_block"): (40.28e6, "fused_block.cuh", "6a4e4ced52da"),
    ("swin_b_s1", "fused_block"): (59.91e6, "fused_block.cuh", "6a4e4ced52da"),
    ("swinv2_t_s1", "fused_block"): (25.38e6, "fused_block.cuh", "6a4e4ced52da"),
    ("swinv2_l_w24", "window_attention"): (896.15e6, "attn_window.cu", "4cd6a274a957"),
    # (q|k|v, 38.5 MB, stays in L2 for the attention kernel: DRAM sees x and the weights)
    ("swin_b_s3", "qkv_gemm"): (14.52e6, "gemm_tc.cu", "81cba03b5e19"),
}


def profiled_traffic(workload, kernel):
    import hashlib
    ent = PROFILED_TRAFFIC.get((workload, kernel))
    if not ent:
        return None
    path = os.path.join(ROOT, "vision_transformer_shifted_gb300", "csrc", ent[1])
    try:
        sha = hashlib.sha1(open(path, "rb").read()).hexdigest()[:12]
    except OSError:
        return None
    return ent[0] if sha == ent[2] else None
METRIC = "fused shifted-window attn block tokens/s & TFLOP/s; % of bf16/HBM roofline"
# the workloads of the 'configs' record, in their order of definition
CONFIG_KEYS = ["tiny", "swin_t_s1", "swin_b_s1", "swin_b_s3", "swinv2_t_s1", "swinv2_l_w24"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sust=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus, backend=None):
    """(rank, world, local rank, torch.distributed or None) from the torchrun
    environment; NCCL on GPUs, gloo where there is none (the CPU tests)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
        if not dist.is_initialized():
            dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(v, dist):
    if dist is None:
        return v
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(w, rank):
    """Each rank's own batch: the same shapes, its own seed (weak scaling)."""
    return w.with_(seed=w.seed + rank)


def job_rate(tokens_per_rank, world, seconds):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / seconds


def oracle_sample_rate(w, g, table_np, seconds=10.0, threads=None):
    """Tokens/s of the float64 oracle on a bounded sample of windows."""
    import oracle
    a = {k: (v.double().numpy() if v is not None else None) for k, v in g.items()}
    threads = threads or len(os.sched_getaffinity(0))
    rng = np.random.default_rng(0)
    n = max(threads, 4)
    done_windows, elapsed = 0, 0.0
    while elapsed < seconds:
        wins = rng.integers(0, w.n_windows, size=n)
        t0 = time.perf_counter()
        oracle.forward(a["x"], a["Wqkv"], a["bqkv"], table_np, a.get("tau"), a["Wproj"], a["bproj"],
                       heads=w.heads, M=w.M, shift=w.shift, mode=w.mode, windows=wins, nthreads=threads)
        dt = time.perf_counter() - t0
        done_windows += n
        elapsed += dt
        if dt < seconds / 8:
            n *= 2
    return done_windows * w.N / elapsed, threads, done_windows


def table_for(w, g, dev, h=None):
    """Relative-bias table: V1 draws it; V2 builds it on the GPU with the
    meta-network kernel (swin_wattn_cpb_table), as a user would once."""
    from vision_transformer_shifted_gb300 import binding as sw
    if w.mode != V2:
        return g["table"].to(dev)
    tab = torch.empty(((2 * w.M - 1) ** 2, w.heads), dtype=torch.bfloat16 if w.dtype == "bf16" else torch.float32,
                      device=dev)
    sw.swin_wattn_cpb_table(h, g["W1"].to(dev), g["b1"].to(dev), g["W2"].to(dev), tab)
    return tab


def run_reference(args, w):
    rank, world, local, dist = dist_setup(args.gpus)
    if rank != 0:
        return
    import oracle
    g = generate(w)
    if w.mode == V2:
        table = oracle.cpb_table(g["W1"].double().numpy(), g["b1"].double().numpy(), g["W2"].double().numpy(),
                                 M=w.M, heads=w.heads)
    else:
        table = g["table"].double().numpy()
    per_step = []
    threads = len(os.sched_getaffinity(0))
    # each step is a bounded sample, sized so the whole run stays near 2.5 minutes
    step_s = max(0.2, min(args.ref_seconds, 150.0 / (args.steps + args.warmup)))
    for _ in range(args.warmup + args.steps):
        rate, threads, nw = oracle_sample_rate(w, g, table, seconds=step_s, threads=threads)
        per_step.append(rate)
    rate = statistics.median(per_step[args.warmup:])
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.tokens / rate * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.key, "B": w.B, "H": w.H, "W": w.W, "C": w.C, "heads": w.heads, "M": w.M,
                       "shift": w.shift, "mode": "V2" if w.mode == V2 else "V1"},
            "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": "random windows per step, about %.2f s of float64 CPU work each; "
                                       "tokens/s scaled from the windows done" % step_s},
            "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_forward(sw, w, dev, pk, args, steps, soak, rank=0, world=1, dist=None, path=0):
    """Times `steps` forwards of workload `w` (CUDA events on the launching
    stream, inputs rotated over buffer sets larger than 2x L2), then each
    kernel of the three-kernel path on its own.  Returns a dict of figures and
    the objects the end-to-end leg reuses."""
    mode = w.mode | (sw.FP32 if w.dtype == "fp32" else 0)
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, mode)
    if path:
        sw.swin_wattn_set_option(h, sw.OPT_PATH, path)
    # fixed weights across the steps, as in serving: each step's fused kernel
    # may load them while the step before finishes
    sw.swin_wattn_set_option(h, sw.OPT_OVERLAP_CALLS, args.overlap)
    g = generate(rank_workload(w, rank))
    t = {k: (v.to(dev) if v is not None else None) for k, v in g.items()}
    table = table_for(w, g, dev, h)
    io_bytes = w.tokens * w.C * w.elem_bytes * 2
    nsets = max(2, -(-(2 * L2_BYTES) // io_bytes) + 1)
    xs = [t["x"]] + [torch.randn_like(t["x"], dtype=torch.float32).to(t["x"].dtype) for _ in range(nsets - 1)]
    outs = [torch.empty_like(t["x"]) for _ in range(nsets)]
    stream = torch.cuda.current_stream()

    def step(i):
        k = i % nsets
        sw.swin_wattn_forward(h, xs[k], t["Wqkv"], t["bqkv"], table, t.get("tau"), t["Wproj"], t["bproj"],
                              outs[k], stream)

    for i in range(args.warmup):
        step(i)
    assert sw.swin_wattn_sync_status(h, stream) == sw.OK
    launches_per_step = sw.swin_wattn_last_launches(h)
    # soak (untimed) so that the clock record covers a loaded GPU, then time the steps
    t_soak = time.perf_counter()
    i = 0
    while time.perf_counter() - t_soak < soak:
        step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(e0.elapsed_time(e1), dist) / steps
    # the spread of single steps, from a second pass with an event after every
    # step (outside the timed region above: each event adds about 2 us)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    marks[0].record(stream)
    for i in range(steps):
        step(i)
        marks[i + 1].record(stream)
    torch.cuda.synchronize()
    per_step = sorted(marks[i].elapsed_time(marks[i + 1]) for i in range(steps))
    pct = lambda q: per_step[min(len(per_step) - 1, int(q * (len(per_step) - 1) + 0.5))] * 1e3  # noqa: E731
    assert sw.swin_wattn_sync_status(h, stream) == sw.OK
    tflops = w.flops * world / (ms * 1e-3) / 1e12
    path = ("three kernels" if launches_per_step >= 3 else "fp32 block" if w.dtype == "fp32" else "fused")
    res = {"ms_per_step": ms, "tokens_per_s": job_rate(w.tokens, world, ms * 1e-3), "tflops": tflops,
           "step_us": {"median": pct(0.5), "p10": pct(0.1), "p90": pct(0.9),
                       "note": "second pass, an event after every step (adds about 2 us a step)"},
           "path": path, "launches_per_step": launches_per_step,
           "l2": "inputs rotated over %d buffer sets of %.0f MB (x + out), %.0f MB > 2x L2" %
                 (nsets, io_bytes / 2 ** 20, nsets * io_bytes / 2 ** 20)}
    if w.dtype == "bf16":
        # whole-block roofline: min(dense bf16 peak, HBM x algorithmic intensity)
        ai = w.flops / w.io_bytes
        bound_tf = min(pk["bf16_sust"], pk["hbm"] * 1e9 * ai / 1e12)
        res["block_roofline"] = {"achieved_tflops": tflops / world, "roof_tflops": bound_tf,
                                 "frac": tflops / world / bound_tf, "ai_flop_per_byte": ai,
                                 "algorithmic_bytes": w.io_bytes, "algorithmic_flops": w.flops,
                                 "peak_source": pk["source"] + " (sustained bf16 / copy GB/s)"}
        kernels = {}
        if launches_per_step >= 3:   # the three-kernel path (the QKV GEMM may take several launches)
            kernels = per_kernel_times(sw, h, w, t, table, xs, stream, steps)
        roof = dominant_roofline(w, kernels, pk, ms)
        roof["traffic"] = profiled_traffic(w.key, roof["kernel"])
        if roof["traffic"] is not None:
            # ncu's DRAM counters see what reached DRAM during the launch: output
            # still dirty in L2 when the kernel ends is written back later (and
            # counted for whatever runs then), so traffic can read below the
            # algorithmic bytes; above them it would mean re-reads
            roof["traffic_note"] = ("DRAM bytes read + written during one launch (ncu); output left dirty in "
                                    "L2 at the end is not counted")
        res["roofline"] = roof
        res["kernels_us"] = kernels
    else:
        # the tiny fp32 workload is a correctness case: no roofline
        res["block_roofline"] = None
        res["roofline"] = None
    return res, (h, g, t, table, stream)


def oracle_baseline(w, g, seconds):
    import oracle
    if w.mode == V2:
        tab_np = oracle.cpb_table(g["W1"].double().numpy(), g["b1"].double().numpy(), g["W2"].double().numpy(),
                                  M=w.M, heads=w.heads)
    else:
        tab_np = g["table"].double().numpy()
    rate, threads, nw = oracle_sample_rate(w, g, tab_np, seconds=seconds)
    return {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "%d random windows of this workload (%d tokens), float64, OpenMP over windows" %
                      (nw, nw * w.N)}


def workload_config(w, world):
    return {"workload": w.key, "B": w.B, "H": w.H, "W": w.W, "C": w.C, "heads": w.heads, "M": w.M,
            "shift": w.shift, "mode": "V2" if w.mode == V2 else "V1", "dtype": w.dtype,
            "parallelism": "dp%d (independent batches)" % world}


def run_ours(args, w):
    from vision_transformer_shifted_gb300 import binding as sw
    rank, world, local, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    sw.load()
    pk = peaks()
    with ClockSampler(dev.index) as clk:
        res, (h, g, t, table, stream) = measure_forward(sw, w, dev, pk, args, args.steps, args.soak, rank, world,
                                                        dist, args.path)
    ms = res["ms_per_step"]

    # end to end through the host-buffer entry point (pinned buffers)
    x_host = g["x"].pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    for _ in range(2):
        sw.swin_wattn_forward_host(h, x_host, t["Wqkv"], t["bqkv"], table, t.get("tau"), t["Wproj"], t["bproj"],
                                   out_host, stream)
    torch.cuda.synchronize()
    barrier(dist)
    k_e2e = max(3, args.steps // 4)
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        sw.swin_wattn_forward_host(h, x_host, t["Wqkv"], t["bqkv"], table, t.get("tau"), t["Wproj"], t["bproj"],
                                   out_host, stream)
        stream.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / k_e2e, dist)
    sw.swin_wattn_destroy(h)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(w, g, args.cpu_seconds)

    # every other workload, each in the same way but shorter (one line; not the headline)
    configs = {}
    if args.configs and world == 1:
        for key in CONFIG_KEYS:
            if key == w.key:
                continue
            wk = WORKLOADS[key]
            with ClockSampler(dev.index) as clk_k:
                rk, (hk, gk, *_rest) = measure_forward(sw, wk, dev, pk, args, args.config_steps, 0.3)
            sw.swin_wattn_destroy(hk)
            rk["config"] = workload_config(wk, 1)
            rk["config"]["overlap_calls"] = bool(args.overlap)
            rk["clocks"] = clk_k.summary()
            if not args.no_cpu_baseline:
                rk["cpu_baseline"] = oracle_baseline(wk, gk, args.config_cpu_seconds)
            configs[key] = rk
    if rank != 0:
        return
    cfg = workload_config(w, world)
    cfg.update({"path": res["path"], "l2": res["l2"], "overlap_calls": bool(args.overlap)})
    line = {"metric": METRIC, "value": res["tokens_per_s"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": cfg,
            "tflops": res["tflops"], "step_us": res["step_us"], "block_roofline": res["block_roofline"],
            "roofline": res["roofline"],
            "kernels_us": res.get("kernels_us", {}),
            "cpu_baseline": cpu,
            "e2e": {"value": job_rate(w.tokens, world, e2e_s), "unit": "tokens/s",
                    "h2d_bytes_per_step": w.tokens * w.C * w.elem_bytes,
                    "d2h_bytes_per_step": w.tokens * w.C * w.elem_bytes},
            "gpu_launches": res["launches_per_step"] * args.steps, "clocks": clk.summary()}
    if configs:
        line["configs"] = configs
    print(json.dumps(line), flush=True)


def per_kernel_times(sw, h, w, t, table, xs, stream, steps):
    """Average duration (us) of each kernel of the three-kernel path, timed
    with CUDA events on the launching stream over `steps` launches."""
    qkv = torch.empty(w.tokens, 3 * w.C, dtype=torch.bfloat16, device=xs[0].device)
    attn = torch.empty(w.tokens, w.C, dtype=torch.bfloat16, device=xs[0].device)
    out = torch.empty_like(xs[0])
    n = len(xs)
    res = {}
    stages = {
        "qkv_gemm": lambda i: sw.swin_wattn_test_qkv(h, xs[i % n], t["Wqkv"], t["bqkv"], qkv, stream),
        "window_attention": lambda i: sw.swin_wattn_test_attn(h, qkv, w.B, w.H, w.W, table, t.get("tau"), attn,
                                                              stream),
        "proj_gemm": lambda i: sw.swin_wattn_test_proj(h, attn, w.B, w.H, w.W, t["Wproj"], t["bproj"], out,
                                                       stream),
    }
    for name, fn in stages.items():
        for i in range(3):
            fn(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / steps * 1e3
    return res


def dominant_roofline(w, kernels, pk, ms):
    """Roofline of the kernel that takes the most time: its algorithmic bytes
    (its own inputs and outputs, read or written once) or FLOPs per launch
    over its measured duration."""
    T, C, e = w.tokens, w.C, w.elem_bytes
    wb = lambda rows: rows * C * e  # noqa: E731
    model = {
        # name: (flops, bytes)
        "qkv_gemm": (6 * T * C * C, wb(T) + 3 * wb(T) + 3 * C * C * e),
        "window_attention": (4 * T * w.N * C, 3 * wb(T) + wb(T)),
        "proj_gemm": (2 * T * C * C, wb(T) + wb(T) + C * C * e),
        "fused_block": (w.flops, w.io_bytes),
    }
    if not kernels:
        kernels = {"fused_block": ms * 1e3}
    name = max(kernels, key=kernels.get)
    flops, nbytes = model[name]
    us = kernels[name]
    ai = flops / nbytes
    ridge = pk["bf16"] * 1e12 / (pk["hbm"] * 1e9)
    if ai < ridge:
        ach = nbytes / (us * 1e-6) / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": ach, "peak": pk["hbm"], "unit": "GB/s",
                "frac": ach / pk["hbm"], "traffic": None, "us_per_launch": us, "algorithmic_bytes": nbytes,
                "peak_source": pk["source"] + " copy bandwidth"}
    ach = flops / (us * 1e-6) / 1e12
    return {"kernel": name, "bound": "tensor", "achieved": ach, "peak": pk["bf16"], "unit": "TFLOP/s",
            "frac": ach / pk["bf16"], "traffic": None, "us_per_launch": us, "algorithmic_flops": flops,
            "peak_source": pk["source"] + " bf16 burst"}


def run_block(args, w, ratio=4):
    """The whole Swin block (LayerNorm, attention, residuals, MLP) on workload
    ``w``, one JSON line; not the headline (that is the attention block)."""
    from vision_transformer_shifted_gb300 import binding as sw
    from vision_transformer_shifted_gb300.inputs import generate_block
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sw.load()
    pk = peaks()
    g = generate_block(w, ratio)
    t = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    h_attn = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
    table = table_for(w, g, dev, h_attn)
    sw.swin_wattn_destroy(h_attn)
    params = dict(ln1_gamma=t["ln1_gamma"], ln1_beta=t["ln1_beta"], Wqkv=t["Wqkv"], bqkv=t["bqkv"], bias_table=table,
                  logit_scale=t.get("tau"), Wproj=t["Wproj"], bproj=t["bproj"], ln2_gamma=t["ln2_gamma"],
                  ln2_beta=t["ln2_beta"], W1=t["mlp_W1"], b1=t["mlp_b1"], W2=t["mlp_W2"], b2=t["mlp_b2"])
    h = sw.swin_block_create(w.C, w.heads, w.M, w.shift, w.mode, ratio)
    sw.swin_block_set_option(h, sw.BLOCK_OPT_OVERLAP_CALLS, args.overlap)   # fixed weights across steps
    io_bytes = w.tokens * w.C * 2 * 2
    nsets = max(2, -(-(2 * L2_BYTES) // io_bytes) + 1)
    xs = [t["x"]] + [torch.randn_like(t["x"], dtype=torch.float32).to(t["x"].dtype) for _ in range(nsets - 1)]
    outs = [torch.empty_like(t["x"]) for _ in range(nsets)]
    stream = torch.cuda.current_stream()

    def step(i):
        sw.swin_block_forward(h, xs[i % nsets], params, outs[i % nsets], stream)

    for i in range(args.warmup):
        step(i)
    assert sw.swin_block_sync_status(h, stream) == sw.OK
    with ClockSampler(dev.index) as clk:
        t_soak = time.perf_counter()
        i = 0
        while time.perf_counter() - t_soak < args.soak:
            step(i)
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    assert sw.swin_block_sync_status(h, stream) == sw.OK
    launches = sw.swin_block_last_launches(h)
    sw.swin_block_destroy(h)
    T, C = w.tokens, w.C
    flops = w.flops + 4 * T * C * ratio * C
    alg_bytes = 2 * T * C * 2 + (4 * C * C + 2 * ratio * C * C) * 2
    ai = flops / alg_bytes
    roof_tf = min(pk["bf16_sust"], pk["hbm"] * 1e9 * ai / 1e12)
    tflops = flops / (ms * 1e-3) / 1e12
    line = {"metric": "swin block forward (LayerNorm, shifted-window attention, residuals, MLP) tokens/s",
            "value": T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.key, "B": w.B, "H": w.H, "W": w.W, "C": C, "heads": w.heads, "M": w.M,
                       "shift": w.shift, "mode": "V1 pre-norm" if w.mode == V1 else "V2 residual post-norm",
                       "mlp_ratio": ratio, "overlap_calls": bool(args.overlap)},
            "tflops": tflops,
            "block_roofline": {"achieved_tflops": tflops, "roof_tflops": roof_tf, "frac": tflops / roof_tf,
                               "ai_flop_per_byte": ai, "algorithmic_bytes": alg_bytes, "algorithmic_flops": flops,
                               "peak_source": pk["source"] + " (sustained bf16 / copy GB/s)"},
            "gpu_launches": launches * args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_stage(args, w, depth, ratio=4):
    """A whole stage on workload ``w``'s grid: ``depth`` blocks with shifts
    0, M/2, 0, ... and the merging step (2x2 -> 2C channels); one JSON line."""
    from vision_transformer_shifted_gb300 import binding as sw
    from vision_transformer_shifted_gb300.inputs import generate_block
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sw.load()
    blocks = []
    for i in range(depth):
        wi = w.with_(shift=0 if i % 2 == 0 else w.M // 2, seed=w.seed + 17 * i)
        g = generate_block(wi, ratio)
        t = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
        h_attn = sw.swin_wattn_create(w.C, w.heads, w.M, wi.shift, w.mode)
        table = table_for(wi, g, dev, h_attn)
        sw.swin_wattn_destroy(h_attn)
        params = dict(ln1_gamma=t["ln1_gamma"], ln1_beta=t["ln1_beta"], Wqkv=t["Wqkv"], bqkv=t["bqkv"],
                      bias_table=table, logit_scale=t.get("tau"), Wproj=t["Wproj"], bproj=t["bproj"],
                      ln2_gamma=t["ln2_gamma"], ln2_beta=t["ln2_beta"], W1=t["mlp_W1"], b1=t["mlp_b1"],
                      W2=t["mlp_W2"], b2=t["mlp_b2"])
        blocks.append((sw.swin_block_create(w.C, w.heads, w.M, wi.shift, w.mode, ratio), params, t["x"]))
        sw.swin_block_set_option(blocks[-1][0], sw.BLOCK_OPT_OVERLAP_CALLS, args.overlap)
    gm = torch.Generator().manual_seed(w.seed + 555)
    gam = (1 + 0.1 * torch.randn(4 * w.C, generator=gm)).bfloat16().to(dev)
    bet = (0.1 * torch.randn(4 * w.C, generator=gm)).bfloat16().to(dev)
    Wm = (torch.randn(2 * w.C, 4 * w.C, generator=gm) * (4 * w.C) ** -0.5).bfloat16().to(dev)
    # V2's extra LayerNorm after every `extra_norm`-th block (0: none)
    en_gam = (1 + 0.1 * torch.randn(w.C, generator=gm)).bfloat16().to(dev)
    en_bet = (0.1 * torch.randn(w.C, generator=gm)).bfloat16().to(dev)
    hm = sw.swin_merge_create(w.C)
    x0 = blocks[0][2]
    bufs = [torch.empty_like(x0) for _ in range(2)]
    out = torch.empty(w.B, w.H // 2, w.W // 2, 2 * w.C, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step(_):
        cur = x0
        for i, (h, params, _x) in enumerate(blocks):
            sw.swin_block_forward(h, cur, params, bufs[i % 2], stream)
            cur = bufs[i % 2]
            if args.extra_norm and (i + 1) % args.extra_norm == 0:
                sw.swin_stage_norm(cur, en_gam, en_bet, cur, stream)
        sw.swin_merge_forward(hm, cur, gam, bet, Wm, out, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < args.soak:
            step(0)
            torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    # per step: each block's launches, the extra LayerNorms, the merging step (LayerNorm + GEMM)
    launches = sum(sw.swin_block_last_launches(h) for h, _p, _x in blocks) + 2
    launches += (len(blocks) // args.extra_norm) if args.extra_norm else 0
    for h, _p, _x in blocks:
        assert sw.swin_block_sync_status(h, stream) == sw.OK
        sw.swin_block_destroy(h)
    sw.swin_merge_destroy(hm)
    line = {"metric": "swin stage forward (%d blocks + merging) tokens/s" % depth, "value": w.tokens / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.key, "B": w.B, "H": w.H, "W": w.W, "C": w.C, "heads": w.heads, "M": w.M,
                       "depth": depth, "extra_norm_every": args.extra_norm,
                       "mode": "V1 pre-norm" if w.mode == V1 else "V2 residual post-norm",
                       "mlp_ratio": ratio, "overlap_calls": bool(args.overlap),
                       "l2": "not flushed: one input set (the stage's own intermediates, "
                       "%.0f MB per block, exceed L2)" % (w.tokens * w.C * (3 + ratio) * 2 / 1e6)},
            "gpu_launches": launches * args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)

def run_backward(args, w):
    """Gradients of the attention block (recompute of q, k, v and o, then the
    backward; V2 also the tau gradient) on workload ``w``; one JSON line, not
    the headline."""
    from vision_transformer_shifted_gb300 import binding as sw
    from vision_transformer_shifted_gb300.inputs import generate
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sw.load()
    pk = peaks()
    g = generate(w, nonzero_bias=True)
    t = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    T, C, N, L = w.tokens, w.C, w.N, 2 * w.M - 1
    h = sw.swin_wattn_create(C, w.heads, w.M, w.shift, w.mode)
    sw.swin_wattn_set_option(h, sw.OPT_OVERLAP_CALLS, args.overlap)   # the backward's own kernels
    table = table_for(w, g, dev, h)
    dtau = torch.empty(w.heads, device=dev, dtype=torch.float32) if w.mode == V2 else None
    io_bytes = T * C * 2 * 3
    nsets = max(2, -(-(2 * L2_BYTES) // io_bytes) + 1)
    gen = torch.Generator(device=dev).manual_seed(9)
    xs = [t["x"]] + [torch.randn(t["x"].shape, generator=gen, device=dev).bfloat16() for _ in range(nsets - 1)]
    dys = [torch.randn(t["x"].shape, generator=gen, device=dev).bfloat16() for _ in range(nsets)]
    dxs = [torch.empty_like(t["x"]) for _ in range(nsets)]
    f32 = dict(device=dev, dtype=torch.float32)
    grads = [torch.empty(3 * C, C, **f32), torch.empty(3 * C, **f32), torch.empty(L * L, w.heads, **f32),
             torch.empty(C, C, **f32), torch.empty(C, **f32)]
    stream = torch.cuda.current_stream()

    def step(i):
        k = i % nsets
        sw.swin_wattn_backward(h, xs[k], t["Wqkv"], t["bqkv"], table, t["Wproj"], t["bproj"], dys[k], dxs[k],
                               *grads, logit_scale=t.get("tau"), dlogit_scale=dtau, stream=stream)

    for i in range(args.warmup):
        step(i)
    assert sw.swin_wattn_sync_status(h, stream) == sw.OK
    with ClockSampler(dev.index) as clk:
        t_soak = time.perf_counter()
        i = 0
        while time.perf_counter() - t_soak < args.soak:
            step(i)
            i += 1
            if i % 16 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    assert sw.swin_wattn_sync_status(h, stream) == sw.OK
    launches = sw.swin_wattn_backward_launches(h)
    sw.swin_wattn_destroy(h)
    # recompute: QKV GEMM 6TC^2, logits and P.V 4TNC; backward: do and dWproj
    # 4TC^2, attention (S again, dP, dq, dk, dv) 10TNC, dx and dWqkv 12TC^2
    flops = 22 * T * C * C + 14 * T * N * C
    line = {"metric": "swin window-attention backward (%s, with recompute) tokens/s" % ("V2" if w.mode == V2 else "V1"),
            "value": T / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.key, "B": w.B, "H": w.H, "W": w.W, "C": C, "heads": w.heads, "M": w.M,
                       "shift": w.shift, "l2": "%d input sets of x and dy (%.0f MB each) in rotation" % (
                           nsets, io_bytes / 1e6), "overlap_calls": args.overlap},
            "tflops": flops / (ms * 1e-3) / 1e12, "algorithmic_flops": flops, "gpu_launches": launches * args.steps,
            "peak_source": pk["source"], "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="swin_t_s1", choices=sorted(WORKLOADS))
    ap.add_argument("--batch", type=int, default=0, help="images per step (0: the workload's own batch)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 three kernels, 2 fused")
    ap.add_argument("--overlap", type=int, default=1, choices=[0, 1],
                    help="1: successive forwards overlap (fixed weights; SWIN_WATTN_OPT_OVERLAP_CALLS)")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed load before timing")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=3.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", type=int, default=1,
                    help="1: also time every other workload (shorter), in a 'configs' key of the line")
    ap.add_argument("--config-steps", type=int, default=30)
    ap.add_argument("--config-cpu-seconds", type=float, default=3.0)
    ap.add_argument("--block", action="store_true",
                    help="time the whole Swin block (LayerNorm, attention, residuals, MLP) instead")
    ap.add_argument("--stage", type=int, default=0,
                    help="time a whole stage of this many blocks (alternating shifts) plus the merging step instead")
    ap.add_argument("--extra-norm", type=int, default=0,
                    help="with --stage: V2's extra LayerNorm on the main branch after every this many blocks")
    ap.add_argument("--backward", action="store_true",
                    help="time the gradients of the attention block (with recompute) instead")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.batch > 0 and args.batch != w.B:
        # another batch is another workload: it carries its own name (and no
        # profiled traffic figure)
        w = w.with_(B=args.batch, key="%s_b%d" % (w.key, args.batch))
    if args.stage > 0:
        if w.dtype != "bf16" or args.impl != "ours" or args.gpus != 1 or (w.H // 2) % 1:
            ap.error("--stage: bf16 workloads, our implementation, one GPU")
        run_stage(args, w, args.stage)
    elif args.backward:
        if w.dtype != "bf16" or args.impl != "ours" or args.gpus != 1:
            ap.error("--backward: bf16 workloads, our implementation, one GPU")
        run_backward(args, w)
    elif args.block:
        if w.dtype != "bf16" or args.impl != "ours" or args.gpus != 1:
            ap.error("--block: bf16 workloads, our implementation, one GPU")
        run_block(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
