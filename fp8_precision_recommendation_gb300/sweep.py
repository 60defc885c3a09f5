"""Measured variant table for loka_dispatch_select (LoKA Dispatch).

"LoKA: Low-precision Kernel Applications for Recommendation Models at
Scale", section III-C "Library and Recipe Selection": every candidate recipe
is timed on the layer's shape and its error is measured by the probe; the
selector then keeps the candidates whose error is within budget (and whose
speedup over the high-precision path clears a floor) and picks the fastest.
Section III-A "Offline Error Quantification" measures the error on the
layer's own data; here seeded synthetic activations of the pages' kind stand
in (normal, optionally with 1% of the entries scaled by 100).

The candidates are this library's variants of ``loka_fp8_linear_norm``:
per-tensor, per-row, MX 1x32 and square 32x32-block E4M3 scaling, and the
bf16 path.  For each
problem (M, N, K, norm, outlier fraction) and variant:

* time: the device time of repeated calls (captured in a CUDA graph and
  replayed under CUDA events on one stream after warm-up), with bf16 X
  quantized inside every call and W quantized once beforehand (model weights
  are static); small problems stay in L2 between calls, which favours every
  variant alike;
* error: ``loka_quant_error`` -- normwise relative error and MERE of the
  pre-norm FP8 output against the same layer on bf16 inputs with fp32
  accumulation, which is the bf16 variant itself (so its error is 0).

Each row is (M, N, K, norm, outlier_frac, variant, time_us, rel_err, mere),
the record that ``dispatch_select`` and the C call take.

Usage (one GPU):
    python -m fp8_precision_recommendation_gb300.sweep --out table.json
    python -m fp8_precision_recommendation_gb300.sweep --quick --out small.json
"""
from __future__ import annotations

import argparse
import json
import math
import os
import time
from typing import Dict, List, Sequence, Tuple

from . import _loka
from . import (LOKA_BF16, LOKA_NORM_LAYER, LOKA_SCALE_BLOCK32, LOKA_SCALE_MX32, LOKA_SCALE_ROW, LOKA_SCALE_TENSOR,
               Layer, Workspace, fp8_linear_norm, quant_error, quantize_fp8)

VARIANTS = (LOKA_SCALE_TENSOR, LOKA_SCALE_ROW, LOKA_SCALE_MX32, LOKA_BF16, LOKA_SCALE_BLOCK32)
# the pages' sweep: M = 4096 .. 524288 in powers of two, K and N from 64 to
# 2048, with and without 1% of the entries of X scaled by 100
GRID_M = tuple(4096 << i for i in range(8))
GRID_K = (64, 128, 256, 512, 1024, 2048)
GRID_N = (64, 128, 256, 512, 1024, 2048)
OUTLIERS = (0.0, 0.01)

Row = Tuple[int, int, int, int, float, int, float, float, float]


def problems(quick: bool = False) -> List[Tuple[int, int, int, int, float]]:
    """(M, N, K, norm, outlier_frac) of the sweep grid."""
    if quick:
        return [(4096, 64, 128, LOKA_NORM_LAYER, 0.0), (4096, 256, 512, LOKA_NORM_LAYER, 0.01)]
    return [(m, n, k, LOKA_NORM_LAYER, o) for m in GRID_M for k in GRID_K for n in GRID_N for o in OUTLIERS]


def synthetic_layer(M: int, N: int, K: int, outlier_frac: float, seed: int, device):
    """Seeded device-side draw: X ~ N(0,1) with a Bernoulli(outlier_frac)
    mask of entries times 100, W ~ N(0, 1/K), bias ~ N(0, 0.02); bf16."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0:
        mask = torch.rand((M, K), generator=g, device=device) < outlier_frac
        x = torch.where(mask, x * 100.0, x)
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * (1.0 / math.sqrt(K))
    b = torch.randn((N,), generator=g, device=device, dtype=torch.float32) * math.sqrt(0.02)
    return x.to(torch.bfloat16), w.to(torch.bfloat16), b.to(torch.bfloat16)


def time_call(fn, stream, min_ms: float = 2.0, warmup: int = 3) -> float:
    """Mean microseconds per call of the device work: the calls are captured
    in a CUDA graph (so the host's cost per call is not in the time) and the
    graph replayed under CUDA events on `stream`, with enough calls in it to
    cover at least `min_ms`."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        reps = 1
        while True:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                for _ in range(reps):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b)
            del g
            if ms >= min_ms or reps >= 1024:
                return 1e3 * ms / reps
            reps *= 2


def measure(M: int, N: int, K: int, norm: int, outlier_frac: float, seed: int = 0,
            variants: Sequence[int] = VARIANTS) -> List[Row]:
    """Rows of every supported variant for one problem."""
    import torch
    dev = torch.device("cuda")
    stream = torch.cuda.Stream()
    ws = Workspace(dev)
    x, w, bias = synthetic_layer(M, N, K, outlier_frac, seed, dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    # the draw ran on the current stream; the measurements run on `stream`
    stream.wait_stream(torch.cuda.current_stream())
    rows: List[Row] = []
    for v in variants:
        try:
            if v == LOKA_BF16:
                layer = Layer(x=x, w=w, bias=bias, mode=v, norm=norm, eps=1e-5, y=y)
                err = {"rel_err_fro": 0.0, "mere": 0.0}
            else:
                qw, sw = quantize_fp8(w, v, workspace=ws, stream=stream.cuda_stream)
                layer = Layer(x=x, w=qw, w_scales=sw, bias=bias, mode=v, norm=norm, eps=1e-5, y=y)
                err = quant_error(x, w, bias, v, workspace=ws, stream=stream.cuda_stream)
            t = time_call(lambda: fp8_linear_norm([layer], workspace=ws, stream=stream.cuda_stream), stream)
        except _loka.LokaError as e:
            if e.status == _loka.LOKA_ERR_UNSUPPORTED:
                continue
            raise
        rows.append((M, N, K, norm, outlier_frac, v, t, float(err["rel_err_fro"]), float(err["mere"])))
    return rows


def run(quick: bool = False, log=print) -> Dict:
    import torch
    rows: List[Row] = []
    t0 = time.time()
    for i, (m, n, k, norm, o) in enumerate(problems(quick)):
        got = measure(m, n, k, norm, o, seed=i)
        rows.extend(got)
        log(f"M={m} N={n} K={k} outliers={o}: " +
            ", ".join(f"v{r[5]} {r[6]:.1f}us err {r[7]:.2e}" for r in got))
        torch.cuda.empty_cache()
    return {"device": torch.cuda.get_device_name(), "seconds": round(time.time() - t0, 1),
            "columns": ["M", "N", "K", "norm", "outlier_frac", "variant", "time_us", "rel_err", "mere"],
            "variants": {"0": "per-tensor E4M3", "1": "per-row E4M3", "2": "MX 1x32 E4M3/E8M0", "3": "bf16",
                         "4": "square 32x32 E4M3/E8M0"},
            "rows": [list(r) for r in rows]}


def load_table(path: str) -> List[Row]:
    """Rows of a table written by run(), as dispatch_select takes them."""
    with open(path) as f:
        d = json.load(f)
    return [tuple(r) for r in d["rows"]]


DEFAULT_TABLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "dispatch_table_gb300.json")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--out", default=DEFAULT_TABLE)
    ap.add_argument("--quick", action="store_true", help="two small problems (a smoke run)")
    args = ap.parse_args()
    table = run(quick=args.quick)
    with open(args.out, "w") as f:
        json.dump(table, f, indent=0)
    print(f"{len(table['rows'])} rows -> {args.out} ({table['seconds']} s)")


if __name__ == "__main__":
    main()
