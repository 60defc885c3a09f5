"""FP8 GEMM, dequantization + bias, LayerNorm / RMSNorm, bf16 output.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What one layer computes (LoKA page, section II-C: the FP8 linear y = Wx + b;
section III-B "Block-wise Normalization": the normalization that follows the
GEMM on the same output row; RMSNorm and LayerNorm as named there):

  acc[m,n] = sum_k decode(qx[m,k]) * decode(qw[n,k])            (exact)
  v[m,n]   = acc[m,n] * sx[m] * sw[n] + b[n]                     (tensor/row)
  v[m,n]   = sum_k decode(qx)*2^ex[m,k/32] * decode(qw)*2^ew[n,k/32] + b[n] (MX)
             (square 32x32 blocks: the exponents are ex[m/32,k/32], ew[n/32,k/32])
  v[m,n]   = sum_k x[m,k] * w[n,k] + b[n]                        (BF16 path)
  LayerNorm: y = (v - mean_n v) / sqrt(var_n v + eps) * gamma + beta
             (biased variance, 1/N)
  RMSNorm:   y = v / sqrt(mean_n v^2 + eps) * gamma
  BlockNorm: the RMSNorm of each block of `norm_block` consecutive columns
             of a row, then * gamma (section III-B 2: RMSNorm applied to
             (Wx + b).view(-1, BlockN), a grouped RMSNorm)
  Hard Swish (optional, after the norm; section III-B 3):
             y * ReLU6(y + 3) / 6
  out = bf16(y), round to nearest even from float64.

The GEMM is taken in float64.  For tensorwise and rowwise scaling every
product decode(qx)*decode(qw) is a multiple of 2^-18 no larger than 448^2 <
2^18, so any partial sum over K <= 2^16 terms needs fewer than 53 bits and
the float64 matmul is exact whatever order the library sums in.
"""
from __future__ import annotations

import numpy as np
import torch

from .formats import bf16_round, e4m3_decode, e8m0_decode
from .quantize import as_f32, quantize, MX_BLOCK

SCALE_TENSOR, SCALE_ROW, SCALE_MX32, SCALE_BF16, SCALE_BLOCK32 = 0, 1, 2, 3, 4
NORM_NONE, NORM_LAYER, NORM_RMS, NORM_BLOCK_RMS = 0, 1, 2, 3
ACT_NONE, ACT_HARDSWISH = 0, 1


def vec64(t, n: int, default: float) -> np.ndarray:
    """Optional bf16 parameter vector -> float64 (default value when None)."""
    if t is None:
        return np.full(n, default, dtype=np.float64)
    return as_f32(t).astype(np.float64)


def dequantize(q: np.ndarray, scales, mode: int) -> np.ndarray:
    """decode(q) times its scale, in float64 (exact: scales are applied as
    a float64 product of a 4-bit-mantissa value and a float32 scale, or a
    power of two)."""
    vals = e4m3_decode(q)
    if mode == SCALE_TENSOR:
        return vals * np.float64(scales)
    if mode == SCALE_ROW:
        return vals * np.asarray(scales, dtype=np.float64)[:, None]
    if mode == SCALE_MX32:
        f = e8m0_decode(scales)
        return vals * np.repeat(f, MX_BLOCK, axis=1)
    if mode == SCALE_BLOCK32:
        f = e8m0_decode(scales)
        return vals * np.repeat(np.repeat(f, MX_BLOCK, axis=0)[:vals.shape[0]], MX_BLOCK, axis=1)
    raise ValueError(mode)


def gemm_exact(qx: np.ndarray, qw: np.ndarray) -> np.ndarray:
    """acc = decode(qx) @ decode(qw)^T in float64 (exact, see module doc)."""
    return e4m3_decode(qx) @ e4m3_decode(qw).T


def prenorm(x, w, bias, mode: int):
    """The linear output v = (scaled FP8 GEMM) + b before normalization.

    Returns (v float64 [M,N], quantized operands as a dict).
    """
    N = w.shape[0]
    b = vec64(bias, N, 0.0)
    if mode == SCALE_BF16:
        v = as_f32(x).astype(np.float64) @ as_f32(w).astype(np.float64).T
        return v + b[None, :], {}
    qx, sx = quantize(x, mode)
    qw, sw = quantize(w, mode)
    if mode in (SCALE_MX32, SCALE_BLOCK32):
        v = dequantize(qx, sx, mode) @ dequantize(qw, sw, mode).T
    else:
        acc = gemm_exact(qx, qw)
        sxv = np.full(acc.shape[0], np.float64(sx)) if mode == SCALE_TENSOR else sx.astype(np.float64)
        swv = np.full(acc.shape[1], np.float64(sw)) if mode == SCALE_TENSOR else sw.astype(np.float64)
        v = acc * sxv[:, None] * swv[None, :]
    return v + b[None, :], {"qx": qx, "sx": sx, "qw": qw, "sw": sw}


def layernorm(v: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float) -> np.ndarray:
    mu = v.mean(axis=1, keepdims=True)
    var = ((v - mu) ** 2).mean(axis=1, keepdims=True)
    return (v - mu) / np.sqrt(var + eps) * gamma[None, :] + beta[None, :]


def rmsnorm(v: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    ms = (v * v).mean(axis=1, keepdims=True)
    return v / np.sqrt(ms + eps) * gamma[None, :]


def blocknorm(v: np.ndarray, gamma: np.ndarray, eps: float, block: int) -> np.ndarray:
    """RMSNorm of every `block` consecutive columns of each row, then gamma."""
    M, N = v.shape
    assert N % block == 0
    vb = v.reshape(M, N // block, block)
    ms = (vb * vb).mean(axis=2, keepdims=True)
    return (vb / np.sqrt(ms + eps)).reshape(M, N) * gamma[None, :]


def hardswish(y: np.ndarray) -> np.ndarray:
    """h-swish(y) = y * ReLU6(y + 3) / 6, with ReLU6(t) = min(max(t, 0), 6)."""
    return y * np.minimum(np.maximum(y + 3.0, 0.0), 6.0) / 6.0


def normalize(v: np.ndarray, norm: int, gamma, beta, eps: float, norm_block: int = 256) -> np.ndarray:
    N = v.shape[1]
    g = vec64(gamma, N, 1.0)
    if norm == NORM_LAYER:
        return layernorm(v, g, vec64(beta, N, 0.0), eps)
    if norm == NORM_RMS:
        return rmsnorm(v, g, eps)
    if norm == NORM_BLOCK_RMS:
        return blocknorm(v, g, eps, norm_block)
    if norm == NORM_NONE:
        return v
    raise ValueError(norm)


def linear_norm(x, w, bias, gamma, beta, mode: int, norm: int, eps: float, norm_block: int = 256,
                act: int = ACT_NONE):
    """Full layer: returns (y_exact float64, y_bf16 float64, operands)."""
    v, ops = prenorm(x, w, bias, mode)
    y = normalize(v, norm, gamma, beta, eps, norm_block)
    if act == ACT_HARDSWISH:
        y = hardswish(y)
    elif act != ACT_NONE:
        raise ValueError(act)
    return y, bf16_round(y), ops


def _check_row_sample(mode: int, rows) -> None:
    """A row sample computes the same rows as the whole layer when the
    activation scales are row-local (per row, MX, bf16), or, for square 32x32
    blocks, when the sample is made of whole aligned 32-row blocks."""
    if mode == SCALE_TENSOR:
        raise ValueError("per-tensor scaling is not row-local")
    if mode == SCALE_BLOCK32:
        r = np.asarray(rows).reshape(-1)
        ok = r.size % 32 == 0 and all(r[i] % 32 == 0 and np.array_equal(r[i:i + 32], r[i] + np.arange(32))
                                      for i in range(0, r.size, 32))
        if not ok:
            raise ValueError("a 32x32-block sample must be whole aligned 32-row blocks")


def linear_norm_inputs(inp, rows=None):
    """Run ``linear_norm`` on a ``workloads.LayerInputs``.

    ``rows`` (optional index array) restricts the output to those rows.  It is
    only valid for row-local scaling (per row, MX, BF16), where each output row
    depends on its own input row alone; per-tensor scaling needs every row.
    """
    x = inp.x
    if rows is not None:
        _check_row_sample(inp.mode, rows)
        x = inp.x[torch.as_tensor(rows, dtype=torch.long)]
    return linear_norm(x, inp.w, inp.bias, inp.gamma, inp.beta, inp.mode, inp.norm, inp.eps,
                       inp.norm_block, inp.act)


def linear_norm_quantized(x, w, bias, gamma, beta, mode: int, norm: int, eps: float, out_mode: int,
                          norm_block: int = 256, act: int = ACT_NONE):
    """The layer, then the next layer's activation quantization of its output.

    GEM Training page, "Handling Quantization Overhead" (the activation
    quantization of a linear layer fused into the normalization before it)
    and "Low Precision Flash Attention" (the fused kernels emit FP8
    activations with their scale factors).  The layer's output is the bf16
    tensor Y that ``linear_norm`` returns; what the next layer receives is Y
    quantized like any activation (``quantize`` with ``out_mode``, per row or
    MX 1x32 along the output columns).  Reading: the codes come from the bf16
    Y, not from the unrounded normalized values, so the fused path hands the
    next layer the same bytes as the unfused one (store Y, quantize it).

    Returns (y_exact float64, y_bf16 float64, q uint8 [M,N], scales).
    """
    y, yb, _ = linear_norm(x, w, bias, gamma, beta, mode, norm, eps, norm_block, act)
    q, s = quantize(yb.astype(np.float32), out_mode)
    return y, yb, q, np.asarray(s)


def linear_norm_quantized_inputs(inp, out_mode: int, rows=None):
    """``linear_norm_quantized`` on a ``workloads.LayerInputs`` (``rows`` as in
    ``linear_norm_inputs``; row-local for every out_mode this takes)."""
    x = inp.x
    if rows is not None:
        _check_row_sample(inp.mode, rows)
        x = inp.x[torch.as_tensor(rows, dtype=torch.long)]
    return linear_norm_quantized(x, inp.w, inp.bias, inp.gamma, inp.beta, inp.mode, inp.norm, inp.eps, out_mode,
                                 inp.norm_block, inp.act)
