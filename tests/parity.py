"""Acceptance rules shared by the GPU parity tests.

bf16 outputs: per element |gpu - exact| <= 2 bf16 ulps of max(|exact|, floor)
and, after normalization, |gpu - exact| <= 1e-2 beyond the unavoidable bf16
output rounding (half an ulp of the exact value): a LayerNorm row with one
dominant element reaches |y| ~ sqrt(N), where one bf16 ulp alone exceeds 1e-2.  The floor (2^-6 for
normalized outputs, 2^-6 times the row RMS for un-normalized ones) keeps the
ulp criterion meaningful for outputs that cancel to nearly zero, where any
fp32 accumulator carries an absolute, not a relative, error.
"""
import numpy as np
import torch

from oracle.formats import bf16_ulp

ULPS = 2.0
MAX_ABS_POST_NORM = 1e-2


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def check_bf16_output(gpu, y_exact, normalized: bool, what: str = ""):
    g = to64(gpu)
    y = np.asarray(y_exact, dtype=np.float64)
    assert g.shape == y.shape, (g.shape, y.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    if normalized:
        floor = np.full((y.shape[0], 1), 2.0 ** -6)
    else:
        floor = 2.0 ** -6 * np.sqrt(np.mean(y * y, axis=1, keepdims=True))
    tol = ULPS * bf16_ulp(np.maximum(np.abs(y), floor))
    err = np.abs(g - y)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements beyond {ULPS} bf16 ulps; "
                             f"first {[(tuple(k), g[tuple(k)], y[tuple(k)]) for k in i]}")
    if normalized:
        excess = err - bf16_ulp(y) / 2
        assert excess.max() <= MAX_ABS_POST_NORM, f"{what}: error beyond bf16 rounding {excess.max()}"
    return float(err.max()) if err.size else 0.0
