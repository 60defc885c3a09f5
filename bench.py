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
    ap.add_argument("--M", type=int, default=65536, help="rows of X (65536 is the headline workload)")
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
def workload(rank: int, M: int = 65536):
    import workloads as W
    return W.rec_mlp(seed=rank, M=M)


def algorithmic_bytes_step(M, K, N):
    # bf16 X read once, bf16 W read once, bias/gamma/beta, bf16 Y written once
    return 2 * M * K + 2 * N * K + 3 * 2 * N + 2 * M * N


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gemm_norm.cu", "quantize.cu", "ptx.cuh", "loka_internal.h"):
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
    rng = np.random.default_rng(123)
    done, t_total = 0, 0.0
    while t_total < budget_s and done < 64 * rows_per_call:
        start = int(rng.integers(0, max(1, M - rows_per_call)))
        rows = np.arange(start, min(M, start + rows_per_call))
        t0 = time.perf_counter()
        OL.linear_norm_inputs(inp, rows=rows)
        t_total += time.perf_counter() - t0
        done += len(rows)
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
    inp = workload(0, args.M)
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
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"rec_mlp M={M} K={K} N={N} per-row E4M3, LayerNorm",
                                        "sample": f"512 rows of X per step (rows are independent under per-row scaling)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_total} rows in {args.steps} steps of 512 rows"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ours
def run_ours(args, world, rank, local):
    import torch
    import fp8_precision_recommendation_gb300 as loka
    from fp8_precision_recommendation_gb300 import _loka

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _loka.load()
    inp = workload(rank, args.M)
    M, K, N = inp.M, inp.K, inp.N
    flops = 2.0 * M * N * K
    x_bytes = 2 * M * K
    nbuf = max(2, math.ceil(3 * L2_BYTES / (x_bytes + 2 * M * N)))
    xs = [inp.x.to(dev) for _ in range(nbuf)]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    w, bias = inp.w.to(dev), inp.bias.to(dev)
    ws = loka.Workspace(dev)
    stream = torch.cuda.Stream(device=dev)

    def layer(i):
        return loka.Layer(x=xs[i % nbuf], w=w, bias=bias, mode=inp.mode, norm=inp.norm, eps=inp.eps,
                          y=ys[i % nbuf])

    def step(i):
        loka.fp8_linear_norm([layer(i)], workspace=ws, stream=stream.cuda_stream)

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

    # ---- per-kernel timing (same launches, same stream) for the roofline
    kern = {}
    qx = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((M,), dtype=torch.float32, device=dev)
    qw = torch.empty((N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((N,), dtype=torch.float32, device=dev)

    def timed(fn, n):
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(n):
                fn(i)
            b.record(stream)
            b.synchronize()
        return a.elapsed_time(b) / 1e3 / n

    s = stream.cuda_stream
    kern["quantize_x"] = timed(lambda i: _loka.loka_quantize_fp8(xs[i % nbuf], M, K, 1, qx, sx, None, 0, s), args.steps)
    _loka.loka_quantize_fp8(w, N, K, 1, qw, sw, None, 0, s)
    gl = [loka.Layer(x=qx, w=qw, x_scales=sx, w_scales=sw, bias=bias, mode=inp.mode, norm=inp.norm, eps=inp.eps,
                     y=ys[i]) for i in range(nbuf)]
    kern["gemm_norm"] = timed(lambda i: loka.fp8_linear_norm([gl[i % nbuf]], workspace=ws, stream=s), args.steps)
    torch.cuda.synchronize()
    bytes_q = 2 * M * K + M * K + 4 * M
    bytes_g = M * K + 4 * M + N * K + 4 * N + 3 * 2 * N + 2 * M * N
    P, src = peaks()
    bw = P["hbm_gbs"]
    dom = "gemm_norm" if kern["gemm_norm"] >= kern["quantize_x"] else "quantize_x"
    dom_bytes = bytes_g if dom == "gemm_norm" else bytes_q
    achieved = dom_bytes / kern[dom] / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": bw, "unit": "GB/s", "frac": achieved / bw,
                "traffic": recorded_traffic(dom), "kernel": dom, "peak_source": f"{src} hbm_gbs",
                "algorithmic_bytes_per_launch": dom_bytes, "launch_us": kern[dom] * 1e6}
    step_bytes = algorithmic_bytes_step(M, K, N)
    step_time = t / args.steps
    path_roofline = {"bytes_per_step": step_bytes, "floor_us": step_bytes / (bw * 1e9) * 1e6,
                     "frac_of_hbm_floor": (step_bytes / (bw * 1e9)) / step_time,
                     "achieved_gbs": step_bytes / step_time / 1e9}

    # ---- comparators: our bf16 GEMM+norm and torch eager bf16 linear + layer_norm
    compare = {}
    if not args.no_compare:
        bl = [loka.Layer(x=xs[i], w=w, bias=bias, mode=3, norm=inp.norm, eps=inp.eps, y=ys[i]) for i in range(nbuf)]
        compare["loka_bf16_fused_us"] = 1e6 * timed(lambda i: loka.fp8_linear_norm([bl[i % nbuf]], workspace=ws, stream=s), args.steps)

        def torch_bf16(i):
            v = torch.nn.functional.linear(xs[i % nbuf], w, bias)
            torch.nn.functional.layer_norm(v, (N,), eps=inp.eps)
        compare["torch_bf16_linear_layernorm_us"] = 1e6 * timed(torch_bf16, args.steps)
        compare["loka_fp8_step_us"] = 1e6 * step_time

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        hx = inp.x.pin_memory()
        hy = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
        dx = torch.empty_like(xs[0])
        dy = torch.empty_like(ys[0])
        el = loka.Layer(x=dx, w=w, bias=bias, mode=inp.mode, norm=inp.norm, eps=inp.eps, y=dy)

        def e2e_step(i):
            dx.copy_(hx, non_blocking=True)
            loka.fp8_linear_norm([el], workspace=ws, stream=s)
            hy.copy_(dy, non_blocking=True)

        te = timed(e2e_step, max(3, args.steps // 2))
        te = max_over_ranks(world, te, dev)
        e2e = {"value": world * flops / te / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": x_bytes,
               "d2h_bytes_per_step": 2 * M * N}

    cpu = None
    if rank == 0 and not args.no_cpu:
        v, rows, tc = oracle_throughput(inp, 10.0)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
               "sample": f"{rows} rows of X (4096-row slices, per-row scaling is row-local), {tc:.1f} s"}

    status = _loka.loka_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    launches_per_step = 2   # one quantize launch (X and W), one GEMM+norm launch
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_time, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
        "config": {"workload": f"rec_mlp X[{M},{K}] N(0,1)+1%x100 outliers, W[{N},{K}] N(0,1/{K}), per-row E4M3, "
                               f"bias, LayerNorm over {N}, bf16 out", "l2": f"{nbuf} rotating X/Y buffers "
                               f"({nbuf * (x_bytes + 2 * M * N) / 1e6:.0f} MB) > L2", "parallelism": f"rows x{world}",
                   "timing": "CUDA graph of K steps, CUDA events on the launching stream"},
        "roofline": roofline, "path_roofline": path_roofline, "kernels_us": {k: v * 1e6 for k, v in kern.items()},
        "compare": compare, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


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
