#!/usr/bin/env python
"""Throughput of the FP8 linear + LayerNorm layer on GB300.

Default workload: the recommendation MLP layer X[65536,512] (bf16, N(0,1)
with 1% of entries x100) times W[256,512]^T, per-row E4M3 scaling of X and W,
fp32 accumulation, bias, LayerNorm over N=256, bf16 output.  One step is the
whole path on one batch: amax + scale + E4M3 cast of X and W, the FP8 GEMM
and the fused dequant/bias/LayerNorm/store epilogue, through the C ABI.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the plain, unoptimized restatement of the method), on a bounded
sample of the same workload, and prints the same line with impl=reference.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 126 * 1024 * 1024
METRIC = "FP8 linear+LayerNorm TFLOP/s & % roofline at M=65536,K=512,N=256 on 1 GB300"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0   # nominal dense ratio (4.5 / 2.25 PFLOP/s)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-compare", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="default workload only: skip the ensemble / MX layer lines and the tensor-core peak")
    ap.add_argument("--M", type=int, default=None, help="rows of X per layer (default: the workload's own)")
    ap.add_argument("--workload", default="rec_mlp",
                    choices=["rec_mlp", "ensemble", "mxfp8", "single", "wide_blocknorm", "rec_mlp_block32"])
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------- workload
def workload(rank: int, M=None):
    import workloads as W
    return W.rec_mlp(seed=rank, **({"M": M} if M else {}))


def algorithmic_bytes_step(M, K, N):
    # bf16 X read once, bf16 W read once, bias/gamma/beta, bf16 Y written once
    return 2 * M * K + 2 * N * K + 3 * 2 * N + 2 * M * N


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gemm_norm.cuh", "gemm_norm.cu", "gemm_e4m3.cu", "quantize.cu", "quant_math.cuh", "ptx.cuh",
              "loka_internal.h"):
        with open(os.path.join(ROOT, "fp8_precision_recommendation_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel
    source is unchanged since it was taken; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("bytes_per_launch")


# ------------------------------------------------------------ CPU oracle
def oracle_throughput(inp, budget_s: float, rows_per_call: int = 4096):
    """Times the oracle on bounded row samples of the workload (row-local
    per-row scaling, so a row sample is the same computation); returns
    (TFLOP/s, rows processed, seconds)."""
    import numpy as np
    import torch
    from oracle import linear as OL
    M, K, N = inp.M, inp.K, inp.N
    if inp.mode == 0:   # per-tensor scaling is not row-local: time the whole (small) layer
        t0 = time.perf_counter()
        n = 0
        while True:
            OL.linear_norm_inputs(inp)
            n += 1
            if time.perf_counter() - t0 >= max(budget_s, 1e-3) or n >= 1000:
                break
        tt = time.perf_counter() - t0
        return 2.0 * n * M * N * K / tt / 1e12, n * M, tt
    rng = np.random.default_rng(123)
    done, t_total = 0, 0.0
    while True:   # at least one sample, then until the time budget is spent
        start = int(rng.integers(0, max(1, M - rows_per_call))) // 32 * 32   # whole 32-row blocks
        rows = np.arange(start, min(M, start + rows_per_call))
        t0 = time.perf_counter()
        OL.linear_norm_inputs(inp, rows=rows)
        t_total += time.perf_counter() - t0
        done += len(rows)
        if t_total >= budget_s or done >= 64 * rows_per_call:
            break
    return 2.0 * done * N * K / t_total / 1e12, done, t_total


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- ranks
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ reference
def run_reference(args, world, rank):
    if rank != 0:
        return
    layers = workload_layers(args.workload, 0, args.M)
    inp = layers[0]
    M, K, N = inp.M, inp.K, inp.N
    for _ in range(args.warmup):
        oracle_throughput(inp, 0.0, rows_per_call=512)
    t_steps = []
    rows_total = 0
    for _ in range(args.steps):
        _, rows, t = oracle_throughput(inp, 0.0, rows_per_call=512)
        t_steps.append(t)
        rows_total += rows
    t = sum(t_steps)
    value = 2.0 * rows_total * N * K / t / 1e12
    cores = oracle_threads()
    line = {
        "impl": "reference", "metric": METRIC if args.workload == "rec_mlp" and not args.M else
        f"FP8 linear+norm TFLOP/s ({args.workload} {len(layers)}x{M}x{K}x{N}) on 1 GB300", "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{args.workload} M={M} K={K} N={N} (group 0 of {len(layers)})",
                                        "sample": f"512 rows of X per step (rows are independent under per-row scaling)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_total} rows in {args.steps} steps of 512 rows"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ours
def workload_layers(name: str, rank: int, M):
    import workloads as W
    if name == "rec_mlp":
        return [W.rec_mlp(seed=rank, **({"M": M} if M else {}))]
    if name == "ensemble":
        return W.ensemble(seed=rank, **({"M": M} if M else {}))
    if name == "mxfp8":
        return [W.mxfp8(seed=rank, **({"M": M} if M else {}))]
    if name == "single":
        return [W.single(seed=rank)]
    if name == "wide_blocknorm":
        return [W.wide_blocknorm(seed=rank, **({"M": M} if M else {}))]
    if name == "rec_mlp_block32":
        return [W.rec_mlp(seed=rank, mode=W.SCALE_BLOCK32, **({"M": M} if M else {}))]
    raise ValueError(name)


def scale_bytes(mode, rows, cols):
    return {0: 4, 1: 4 * rows, 2: rows * cols // 32, 4: (rows + 31) // 32 * (cols // 32)}.get(mode, 0)


def tensor_peaks(dev, stream, clock_index):
    """Dense tcgen05 throughput measured by the library's own microbenchmark
    (one CTA per SM issuing back-to-back M=128, N=256 MMAs from shared
    memory): E4M3 as a burst (one ~15 ms launch) and sustained (launches
    back to back for about 2 s, clocks sampled), bf16 as a burst (to check
    the microbenchmark against the measured cuBLAS bf16 peak)."""
    import torch
    from fp8_precision_recommendation_gb300 import _loka
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    s = stream.cuda_stream
    out = {"sms": sms, "shape": "M=128 N=256 per MMA, cta_group::1, fp32 accumulation in tensor memory"}

    def run(kind, mmas, launches):
        with torch.cuda.stream(stream):
            _loka.loka_selftest_mma_peak(kind, 4096, s)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(launches):
                _loka.loka_selftest_mma_peak(kind, mmas, s)
            b.record(stream)
            b.synchronize()
        k = 32 if kind == 0 else 16
        return sms * mmas * launches * 2.0 * 128 * 256 * k / (a.elapsed_time(b) / 1e3) / 1e12

    out["e4m3_burst_tflops"] = run(0, 200_000, 1)
    out["bf16_burst_tflops"] = run(1, 200_000, 1)
    with ClockSampler(clock_index) as clk:
        time.sleep(0.2)
        out["e4m3_sustained_tflops"] = run(0, 2_000_000, 14)
    out["sustained_clocks"] = clk.summary()
    if _loka.loka_device_status() != 0:
        raise RuntimeError("tensor-core peak microbenchmark timed out")
    return out


def link_bandwidth(dev):
    """Plain pinned host <-> device copies of 64 MB (CUDA events, best of 5):
    the ceiling of the end-to-end measurement's copies."""
    import torch
    n = 64 << 20
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    res = {}
    for name, dst, src in (("h2d_gbs", d, h), ("d2h_gbs", h, d)):
        best = 0.0
        for _ in range(6):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            b.synchronize()
            best = max(best, n / (a.elapsed_time(b) / 1e3) / 1e9)
        res[name] = best
    res["bytes"] = n
    return res


def run_ours(args, world, rank, local):
    import torch
    from fp8_precision_recommendation_gb300 import _loka
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _loka.load()
    line = measure(args, args.workload, world, rank, local, dev, main=True)
    extra = args.workload == "rec_mlp" and not args.M and not args.no_extra
    if extra:
        # the grouped ensemble and the MX layer, measured the same way (device
        # time of a CUDA graph of steps, rotating buffers past L2), so their
        # step and kernel rooflines are on record beside the headline
        torch.cuda.empty_cache()
        sub = argparse.Namespace(**{**vars(args), "no_e2e": True, "no_cpu": True})
        line["workloads"] = {}
        for name in ("ensemble", "mxfp8"):
            w = measure(sub, name, world, rank, local, dev, main=False)
            line["workloads"][name] = {k: w[k] for k in ("metric", "value", "unit", "ms_per_step", "config",
                                                           "step_roofline", "roofline", "kernels_us", "compare",
                                                           "fp8_chained_layer", "clocks")}
            torch.cuda.empty_cache()
        line["tensor_peak"] = tensor_peaks(dev, torch.cuda.Stream(device=dev), local)
        mx = line["workloads"]["mxfp8"]
        pk = line["tensor_peak"]["e4m3_sustained_tflops"]
        mx["tensor_frac_of_measured_e4m3"] = mx["value"] / pk
        # the block-scaled GEMM alone against the same peak: a contraction
        # of 2 M N K flops, bound by the tensor pipe or by HBM, whichever is
        # nearer (the line's `roofline` gives its HBM fraction)
        flops_mx = mx["value"] * 1e12 * mx["ms_per_step"] * 1e-3   # 2 M N K of one step
        gemm_tflops = flops_mx / (mx["kernels_us"]["gemm_norm"] * 1e-6) / 1e12
        mx["gemm_tensor"] = {"bound": "tensor", "achieved": gemm_tflops, "peak": pk, "unit": "TFLOP/s",
                             "frac": gemm_tflops / pk, "peak_source": "measured e4m3_sustained_tflops"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure(args, name, world, rank, local, dev, main):
    import torch
    import fp8_precision_recommendation_gb300 as loka
    from fp8_precision_recommendation_gb300 import _loka

    layers = workload_layers(name, rank, args.M if main else None)
    mode, norm, eps = layers[0].mode, layers[0].norm, layers[0].eps
    flops = sum(2.0 * l.M * l.N * l.K for l in layers)
    x_bytes = sum(2 * l.M * l.K for l in layers)
    y_bytes = sum(2 * l.M * l.N for l in layers)
    nbuf = max(2, math.ceil(3 * L2_BYTES / (x_bytes + y_bytes)))
    dv = lambda t: None if t is None else t.to(dev)
    xs = [[l.x.to(dev) for l in layers] for _ in range(nbuf)]
    ys = [[torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev) for l in layers] for _ in range(nbuf)]
    ws_, bs_, gs_, bes_ = ([dv(getattr(l, a)) for l in layers] for a in ("w", "bias", "gamma", "beta"))
    wsp = loka.Workspace(dev)
    stream = torch.cuda.Stream(device=dev)
    s = stream.cuda_stream

    def mk(i, x_list=None, mode_=None, **kw):
        return [loka.Layer(x=(x_list or xs[i % nbuf])[gi], w=ws_[gi], bias=bs_[gi], gamma=gs_[gi], beta=bes_[gi],
                           mode=mode if mode_ is None else mode_, norm=norm, eps=eps, y=ys[i % nbuf][gi],
                           norm_block=layers[gi].norm_block, act=layers[gi].act,
                           **{k: v[gi] for k, v in kw.items()}) for gi in range(len(layers))]

    def step(i):
        loka.fp8_linear_norm(mk(i), workspace=wsp, stream=s)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        # capture K steps in one CUDA graph: the timed region is GPU work only
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(args.steps):
                step(i)
        g.replay()
        torch.cuda.synchronize()
    status = _loka.loka_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        e0.record(stream)
        with torch.cuda.stream(stream):
            g.replay()
        e1.record(stream)
        e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    t = e0.elapsed_time(e1) / 1e3
    t = max_over_ranks(world, t, dev)
    value = world * flops * args.steps / t / 1e12
    clocks = clk.summary()

    def timed(fn, n):
        # n calls captured in one CUDA graph and replayed, so the host's cost
        # per call (argument checks, descriptor encoding) is not in the time
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i)
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream, capture_error_mode="thread_local"):
                for i in range(n):
                    fn(i)
            gr.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            gr.replay()
            b.record(stream)
            b.synchronize()
        return a.elapsed_time(b) / 1e3 / n

    # ---- per-kernel timing (same kernels, same stream) for the roofline
    kern = {}
    # E4M3 activations rotate over the same buffer sets as the bf16 ones, so
    # the GEMM timed alone reads them from HBM, not from L2
    qx = [[torch.empty((l.M, l.K), dtype=torch.uint8, device=dev) for l in layers] for _ in range(nbuf)]
    qw = [torch.empty((l.N, l.K), dtype=torch.uint8, device=dev) for l in layers]
    shp = [(loka.scales_shape(l.M, l.K, mode), loka.scales_shape(l.N, l.K, mode)) for l in layers]
    sx = [[torch.empty(a[0], dtype=getattr(torch, a[1]), device=dev) for a, _ in shp] for _ in range(nbuf)]
    sw = [torch.empty(b[0], dtype=getattr(torch, b[1]), device=dev) for _, b in shp]
    qws = torch.empty(max(256, _loka.loka_quantize_fp8_workspace_size(1, 32, mode)), dtype=torch.uint8, device=dev)

    def quantize_x(i):
        b = i % nbuf
        for gi, l in enumerate(layers):
            _loka.loka_quantize_fp8(xs[b][gi], l.M, l.K, l.K, mode, qx[b][gi], sx[b][gi], qws, qws.numel(), s)

    kern["quantize_x"] = timed(quantize_x, args.steps)
    for gi, l in enumerate(layers):
        _loka.loka_quantize_fp8(ws_[gi], l.N, l.K, l.K, mode, qw[gi], sw[gi], qws, qws.numel(), s)
    pre = [mk(i, x_list=qx[i], x_scales=sx[i], w_scales=sw) for i in range(nbuf)]
    for lst in pre:
        for gi, lay in enumerate(lst):
            lay.w = qw[gi]
    kern["gemm_norm"] = timed(lambda i: loka.fp8_linear_norm(pre[i % nbuf], workspace=wsp, stream=s), args.steps)
    torch.cuda.synchronize()

    # ---- the layer inside an FP8 stack: its input arrives as E4M3 codes and
    # scales from the previous layer's epilogue, and it hands its own output
    # to the next layer the same way (quantization fused into the
    # normalization; no bf16 copy).  Against the unfused layer: the GEMM with
    # bf16 output, then the quantizer on that output.
    chained = None
    out_mode = mode if mode in (1, 2) and (mode == 2 or layers[0].N <= 256) else None
    if out_mode is not None and not args.no_compare:
        yq = [[torch.empty((l.M, l.N), dtype=torch.uint8, device=dev) for l in layers] for _ in range(nbuf)]
        ysh = [loka.scales_shape(l.M, l.N, out_mode) for l in layers]
        ysq = [[torch.empty(a[0], dtype=getattr(torch, a[1]), device=dev) for a in ysh] for _ in range(nbuf)]
        ch = [mk(i, x_list=qx[i], x_scales=sx[i], w_scales=sw) for i in range(nbuf)]
        for i, lst in enumerate(ch):
            for gi, lay in enumerate(lst):
                lay.w, lay.y = qw[gi], None
                lay.y_q_mode, lay.y_q_only, lay.y_q, lay.y_q_scales = out_mode, True, yq[i][gi], ysq[i][gi]
        t_chain = timed(lambda i: loka.fp8_linear_norm(ch[i % nbuf], workspace=wsp, stream=s), args.steps)

        def quantize_y(i):
            b = i % nbuf
            for gi, l in enumerate(layers):
                _loka.loka_quantize_fp8(ys[b][gi], l.M, l.N, l.N, out_mode, yq[b][gi], ysq[b][gi], qws, qws.numel(), s)

        t_qy = timed(quantize_y, args.steps)
        bytes_c = sum(l.M * l.K + scale_bytes(mode, l.M, l.K) + l.N * l.K + scale_bytes(mode, l.N, l.K)
                      + 2 * l.N * sum(v is not None for v in (l.bias, l.gamma, l.beta))
                      + l.M * l.N + scale_bytes(out_mode, l.M, l.N) for l in layers)
        bw_c = peaks()[0]["hbm_gbs"]
        chained = {"layer_us": 1e6 * t_chain, "tflops": flops / t_chain / 1e12, "output": {1: "E4M3 per-row",
                   2: "E4M3 MX 1x32"}[out_mode], "algorithmic_bytes": bytes_c,
                   "achieved_gbs": bytes_c / t_chain / 1e9, "frac_of_hbm": bytes_c / t_chain / 1e9 / bw_c,
                   "unfused_us": 1e6 * (kern["gemm_norm"] + t_qy), "quantize_y_us": 1e6 * t_qy}

    # ---- the same step with static weights (W quantized once, as a trained
    # model's weights are): bf16 X quantized in every step, captured in a
    # CUDA graph like the main measurement
    static_w = [mk(i, w_scales=sw) for i in range(nbuf)]
    for lst in static_w:
        for gi, lay in enumerate(lst):
            lay.w = qw[gi]
    with torch.cuda.stream(stream):
        for i in range(3):
            loka.fp8_linear_norm(static_w[i % nbuf], workspace=wsp, stream=s)
        torch.cuda.synchronize()
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream, capture_error_mode="thread_local"):
            for i in range(args.steps):
                loka.fp8_linear_norm(static_w[i % nbuf], workspace=wsp, stream=s)
        g2.replay()
        torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        g2.replay()
        b1.record(stream)
        b1.synchronize()
    static_w_step = b0.elapsed_time(b1) / 1e3 / args.steps
    vec_bytes = lambda l: 2 * l.N * sum(v is not None for v in (l.bias, l.gamma, l.beta))
    bytes_q = sum(3 * l.M * l.K + scale_bytes(mode, l.M, l.K) for l in layers)
    bytes_g = sum(l.M * l.K + scale_bytes(mode, l.M, l.K) + l.N * l.K + scale_bytes(mode, l.N, l.K) + vec_bytes(l)
                  + 2 * l.M * l.N for l in layers)
    P, src = peaks()
    bw = P["hbm_gbs"]
    dom = "gemm_norm" if kern["gemm_norm"] >= kern["quantize_x"] else "quantize_x"
    dom_bytes = bytes_g if dom == "gemm_norm" else bytes_q
    achieved = dom_bytes / kern[dom] / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": bw, "unit": "GB/s", "frac": achieved / bw,
                "traffic": recorded_traffic(dom) if name == "rec_mlp" and not args.M else None,
                "kernel": dom, "peak_source": f"{src} hbm_gbs",
                "algorithmic_bytes_per_launch": dom_bytes, "launch_us": kern[dom] * 1e6}
    step_bytes = sum(algorithmic_bytes_step(l.M, l.K, l.N) for l in layers)
    step_time = t / args.steps
    # the whole step against the HBM floor of the layer it computes (bf16 X
    # and W read once, bf16 Y written once): the fraction the metric's
    # "% roofline" refers to; `roofline` above is the dominant kernel's
    step_roofline = {"bound": "hbm", "bytes_per_step": step_bytes, "floor_us": step_bytes / (bw * 1e9) * 1e6,
                     "frac": (step_bytes / (bw * 1e9)) / step_time, "achieved_gbs": step_bytes / step_time / 1e9,
                     "peak_gbs": bw, "peak_source": f"{src} hbm_gbs"}

    # ---- comparators: our bf16 GEMM+norm and torch eager bf16 linear + norm
    compare = {}
    if not args.no_compare:
        bl = [mk(i, mode_=3) for i in range(nbuf)]
        compare["loka_bf16_fused_us"] = 1e6 * timed(lambda i: loka.fp8_linear_norm(bl[i % nbuf], workspace=wsp,
                                                                                    stream=s), args.steps)

        def torch_bf16(i):
            for gi, l in enumerate(layers):
                v = torch.nn.functional.linear(xs[i % nbuf][gi], ws_[gi], bs_[gi])
                if norm == 1:
                    v = torch.nn.functional.layer_norm(v, (l.N,), gs_[gi], bes_[gi], eps=eps)
                elif norm == 2:
                    v = torch.nn.functional.rms_norm(v, (l.N,), gs_[gi], eps=eps)
                elif norm == 3:
                    nb = l.norm_block
                    v = torch.nn.functional.rms_norm(v.view(-1, nb), (nb,), eps=eps).view(l.M, l.N)
                    if gs_[gi] is not None:
                        v = v * gs_[gi]
                if l.act:
                    torch.nn.functional.hardswish(v)
        compare["torch_bf16_linear_norm_us"] = 1e6 * timed(torch_bf16, args.steps)
        compare["loka_fp8_step_us"] = 1e6 * step_time
        compare["loka_fp8_step_static_w_us"] = 1e6 * static_w_step

    # ---- end to end through the public API with pinned host buffers: every
    # step copies its bf16 X in (pinned host -> device) and its bf16 Y out
    # (device -> pinned host).  Steps are pipelined over two device buffer
    # sets and three streams (H2D, compute, D2H), so step i's input copy
    # overlaps step i-1's compute and step i-2's output copy.
    e2e = None
    if not args.no_e2e:
        nb = 2
        hx = [l.x.pin_memory() for l in layers]
        hy = [torch.empty((l.M, l.N), dtype=torch.bfloat16).pin_memory() for l in layers]
        dxb = [[torch.empty_like(x) for x in xs[0]] for _ in range(nb)]
        dyb = [[torch.empty_like(y) for y in ys[0]] for _ in range(nb)]
        els = []
        for bi in range(nb):
            el = mk(0, x_list=dxb[bi])
            for gi, lay in enumerate(el):
                lay.y = dyb[bi][gi]
            els.append(el)
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(nb)]
        ev_comp = [torch.cuda.Event() for _ in range(nb)]
        ev_out = [torch.cuda.Event() for _ in range(nb)]

        def e2e_step(i):
            bi = i % nb
            s_in.wait_event(ev_comp[bi])              # compute of step i-nb is done with dx[bi]
            with torch.cuda.stream(s_in):
                for a, b in zip(dxb[bi], hx):
                    a.copy_(b, non_blocking=True)
                ev_in[bi].record(s_in)
            stream.wait_event(ev_in[bi])
            stream.wait_event(ev_out[bi])             # output copy of step i-nb is done with dy[bi]
            loka.fp8_linear_norm(els[bi], workspace=wsp, stream=s)
            ev_comp[bi].record(stream)
            s_out.wait_event(ev_comp[bi])
            with torch.cuda.stream(s_out):
                for a, b in zip(hy, dyb[bi]):
                    a.copy_(b, non_blocking=True)
                ev_out[bi].record(s_out)

        n_e2e = max(4, args.steps // 2)
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        s_in.wait_stream(stream)
        for i in range(n_e2e):
            e2e_step(i)
        stream.wait_stream(s_out)
        a1.record(stream)
        a1.synchronize()
        te = a0.elapsed_time(a1) / 1e3 / n_e2e
        te = max_over_ranks(world, te, dev)
        link = link_bandwidth(dev)
        # copies in and out overlap each other and the compute: the slower
        # direction bounds a step
        t_link = max(x_bytes / (link["h2d_gbs"] * 1e9), y_bytes / (link["d2h_gbs"] * 1e9), step_time)
        e2e = {"value": world * flops / te / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": x_bytes,
               "d2h_bytes_per_step": y_bytes, "pipelined": "2 buffer sets, H2D / compute / D2H streams",
               "link": link, "ceiling": world * flops / t_link / 1e12,
               "frac_of_ceiling": (world * flops / te / 1e12) / (world * flops / t_link / 1e12)}

    cpu = None
    if rank == 0 and not args.no_cpu:
        v, rows, tc = oracle_throughput(layers[0], 10.0)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
               "sample": f"{rows} rows of X (4096-row slices, row-local scaling), {tc:.1f} s"}

    status = _loka.loka_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    launches_per_step = (3 if mode == 0 else 1) + 1   # quantize (amax + cast for per-tensor) + GEMM+norm
    l0 = layers[0]
    desc = {"rec_mlp": "rec-MLP X N(0,1)+1%x100 outliers, per-row E4M3, bias, LayerNorm",
            "ensemble": "8-layer ensemble, per-row E4M3, RMSNorm, one grouped launch",
            "mxfp8": "Laplace X, MX 1x32 E8M0 block scaling, LayerNorm",
            "single": "per-tensor E4M3, LayerNorm",
            "wide_blocknorm": "wide layer N(0,1)+1%x100 outliers, per-row E4M3, bias, BlockNorm 256, Hard Swish",
            "rec_mlp_block32": "rec-MLP X N(0,1)+1%x100 outliers, square 32x32-block E4M3/E8M0, bias, LayerNorm"}[
                name]
    metric = METRIC if name == "rec_mlp" and not args.M else \
        f"FP8 linear+norm TFLOP/s ({name} {len(layers)}x{l0.M}x{l0.K}x{l0.N}) on 1 GB300"
    line = {
        "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_time, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
        "config": {"workload": f"{name}: {len(layers)} x X[{l0.M},{l0.K}] W[{l0.N},{l0.K}], {desc}, bf16 out",
                   "l2": f"{nbuf} rotating X/Y buffer sets ({nbuf * (x_bytes + y_bytes) / 1e6:.0f} MB) > L2",
                   "parallelism": f"rows x{world}",
                   "timing": "CUDA graph of K steps (per-kernel figures: a CUDA graph of K launches each), CUDA events on the launching stream"},
        "roofline": roofline, "step_roofline": step_roofline, "kernels_us": {k: v * 1e6 for k, v in kern.items()},
        "compare": compare, "fp8_chained_layer": chained, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
    }
    return line


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
