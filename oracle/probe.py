"""Per-layer quantization-error probe (MERE and normwise relative error).

TEST INFRASTRUCTURE ONLY (see the package docstring).

LoKA page, section II-C "Error Analysis" defines the mean element-wise
relative error of a low-precision output against a high-precision reference
of the same linear layer, averaged over all M x N output elements; section
III-A "Offline Error Quantification" (Fig. 5) applies it per layer, with
loss = MERE(FP8(Wx+b), high-precision(Wx+b)).

Readings (the extracted formula lost its normalizing factor and says nothing
about zero references):
  * MERE = mean over {(m,n): ref[m,n] != 0} of |out - ref| / |ref|; the number
    of excluded zero references is reported beside it.
  * normwise relative error = ||out - ref||_F / ||ref||_F.
  * max_abs = max |out - ref|.
  * max_abs_post_norm = max |Norm(out) - Norm(ref)|: the same two outputs
    after the layer's normalization (and activation, when it has one), the
    quantity the "max-abs after normalization" acceptance bound speaks of.
    Without a normalization or activation it equals max_abs.
  * The reference is the same layer on the bf16 inputs with exact (here
    float64) accumulation; the pages use TF32.
"""
from __future__ import annotations

import numpy as np

from .linear import ACT_HARDSWISH, ACT_NONE, NORM_NONE, SCALE_BF16, hardswish, normalize, prenorm


def mere(out: np.ndarray, ref: np.ndarray):
    """Returns (MERE over non-zero references, number of zero references)."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nz = ref != 0.0
    n = int(nz.sum())
    if n == 0:
        return 0.0, int(ref.size)
    rel = np.abs(out[nz] - ref[nz]) / np.abs(ref[nz])
    return float(rel.sum() / n), int(ref.size - n)


def normwise(out: np.ndarray, ref: np.ndarray) -> float:
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sqrt((ref * ref).sum())
    return float(np.sqrt(((out - ref) ** 2).sum()) / den) if den > 0 else 0.0


def max_abs(out: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(np.asarray(out, np.float64) - np.asarray(ref, np.float64)))) if np.size(ref) else 0.0


def error_stats(out: np.ndarray, ref: np.ndarray) -> dict:
    m, zeros = mere(out, ref)
    return {"mere": m, "rel_err_fro": normwise(out, ref), "max_abs": max_abs(out, ref),
            "zero_ref_count": zeros, "count": int(np.size(ref))}


def quant_error(x, w, bias, mode: int, norm: int = NORM_NONE, gamma=None, beta=None, eps: float = 0.0,
                norm_block: int = 256, act: int = ACT_NONE) -> dict:
    """Probe of one layer: FP8 pre-norm output vs the high-precision one,
    plus the largest difference of the two after the layer's normalization."""
    out, _ = prenorm(x, w, bias, mode)
    ref, _ = prenorm(x, w, bias, SCALE_BF16)
    st = error_stats(out, ref)
    if norm == NORM_NONE and act == ACT_NONE:
        st["max_abs_post_norm"] = st["max_abs"]
        return st

    def post(v):
        y = normalize(v, norm, gamma, beta, eps, norm_block)
        return hardswish(y) if act == ACT_HARDSWISH else y

    st["max_abs_post_norm"] = max_abs(post(out), post(ref))
    return st
