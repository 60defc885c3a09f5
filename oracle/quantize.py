"""Activation / weight quantization to E4M3: amax, scale selection, cast.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Three scaling granularities, as named on the LoKA page (section II-C and the
recipes of section III-C and Table VI: tensorwise, rowwise, blockwise) and on
the GEM Training page ("Low Precision Flash Attention": MXFP8 scale factors
along each GEMM's K dimension):

  * per tensor: one amax over the whole tensor;
  * per row: one amax per row of a row-major [rows, cols] tensor (per token
    for X[M,K], per output channel for W[N,K]);
  * MX 1x32: one amax per block of 32 consecutive elements along K.

Readings of what the pages leave open (listed in the design notes):
  * amax is the exact max of |x| over the group, NaN ignored (IEEE maxNum).
  * per tensor / per row: inv = fl32(448 / amax) and scale = fl32(amax / 448),
    each one float32 division; q = E4M3(fl32(x * inv)), one float32 multiply;
    amax == 0 gives inv = scale = 1.  The dequantized value is decode(q)*scale.
  * MX: the E8M0 shared exponent is e = floor(log2(amax)) - 8 (8 = the largest
    E4M3 exponent, since 448 = 1.75 * 2^8), clamped to [-127, 127], code
    e + 127; a zero block gives code 0.  q = E4M3(x * 2^-e), which is exact
    scaling (a power of two) followed by the one rounding of the cast.
"""
from __future__ import annotations

import numpy as np
import torch

from .formats import e4m3_encode, floor_log2

F32_448 = np.float32(448.0)
MX_BLOCK = 32
E4M3_EMAX = 8


def as_f32(x) -> np.ndarray:
    """bf16 torch tensor (or array) -> float32 numpy, exactly."""
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").to(torch.float32).numpy()
    return np.asarray(x, dtype=np.float32)


def amax(a: np.ndarray, axis=None) -> np.ndarray:
    """Largest |a| over ``axis``; NaNs are ignored unless all are NaN."""
    return np.fmax.reduce(np.abs(a), axis=axis).astype(np.float32) if axis is not None \
        else np.float32(np.fmax.reduce(np.abs(a).ravel()))


def scales_from_amax(am):
    """(inv, scale) float32 pair(s) for tensorwise / rowwise scaling."""
    am = np.asarray(am, dtype=np.float32)
    zero = am == np.float32(0.0)
    safe = np.where(zero, np.float32(1.0), am).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        inv = (F32_448 / safe).astype(np.float32)
        scale = (safe / F32_448).astype(np.float32)
    inv = np.where(zero, np.float32(1.0), inv).astype(np.float32)
    scale = np.where(zero, np.float32(1.0), scale).astype(np.float32)
    return inv, scale


def quantize_tensor(x):
    """Per-tensor scaling. Returns (q uint8 [R,C], scale float32 scalar)."""
    xf = as_f32(x)
    inv, scale = scales_from_amax(amax(xf))
    with np.errstate(invalid="ignore", over="ignore"):
        y = (xf * np.float32(inv)).astype(np.float32)
    return e4m3_encode(y), np.float32(scale)


def quantize_rows(x):
    """Per-row scaling. Returns (q uint8 [R,C], scales float32 [R])."""
    xf = as_f32(x)
    inv, scale = scales_from_amax(amax(xf, axis=1))
    with np.errstate(invalid="ignore", over="ignore"):
        y = (xf * inv[:, None]).astype(np.float32)
    return e4m3_encode(y), scale.astype(np.float32)


def mx_exponent(am) -> np.ndarray:
    """Shared exponent e = clamp(floor(log2 amax) - 8, -127, 127)."""
    return np.clip(floor_log2(am) - E4M3_EMAX, -127, 127)


def quantize_mx(x):
    """MX 1x32 scaling along the last axis.

    Returns (q uint8 [R,C], e8m0 uint8 [R, C/32]).  C must be a multiple of 32.
    """
    xf = as_f32(x)
    R, C = xf.shape
    assert C % MX_BLOCK == 0
    blocks = xf.reshape(R, C // MX_BLOCK, MX_BLOCK)
    e = mx_exponent(amax(blocks, axis=2))
    with np.errstate(invalid="ignore", over="ignore", under="ignore"):
        y = np.ldexp(blocks, (-e)[:, :, None].astype(np.int32)).astype(np.float32)
    q = e4m3_encode(y).reshape(R, C)
    return q, (e + 127).astype(np.uint8)


def quantize_block32(x):
    """Square 32 x 32 blocks: one E8M0 exponent per block of 32 rows by 32
    columns (GEM Training page, "Low Precision Flash Attention": [32, 32]
    block quantization, transpose-invariant, so a tensor and its transpose
    share one quantization).  The exponent rule is the MX one above, on the
    block's amax; a ragged last block row covers the rows that exist.

    Returns (q uint8 [R,C], e8m0 uint8 [ceil(R/32), C/32]).  C must be a
    multiple of 32.
    """
    xf = as_f32(x)
    R, C = xf.shape
    assert C % MX_BLOCK == 0
    RB, CB = (R + MX_BLOCK - 1) // MX_BLOCK, C // MX_BLOCK
    am = np.zeros((RB, CB), dtype=np.float32)
    for rb in range(RB):
        rows = xf[rb * MX_BLOCK:(rb + 1) * MX_BLOCK]
        for cb in range(CB):
            am[rb, cb] = amax(rows[:, cb * MX_BLOCK:(cb + 1) * MX_BLOCK].ravel(), axis=0)
    e = mx_exponent(am)
    e_full = np.repeat(np.repeat(e, MX_BLOCK, axis=0)[:R], MX_BLOCK, axis=1)
    with np.errstate(invalid="ignore", over="ignore", under="ignore"):
        y = np.ldexp(xf, (-e_full).astype(np.int32)).astype(np.float32)
    return e4m3_encode(y), (e + 127).astype(np.uint8)


def quantize(x, mode: int):
    """Dispatch on the scaling mode id (0 tensor, 1 row, 2 MX 1x32, 4 square
    32x32 blocks)."""
    if mode == 0:
        return quantize_tensor(x)
    if mode == 1:
        return quantize_rows(x)
    if mode == 2:
        return quantize_mx(x)
    if mode == 4:
        return quantize_block32(x)
    raise ValueError(f"no FP8 quantization for mode {mode}")
