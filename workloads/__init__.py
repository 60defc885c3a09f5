"""Seeded synthetic inputs for the FP8 linear + normalization layer.

This module only draws random numbers and rounds them to bf16 storage; it holds
none of the method's arithmetic (no quantization, no GEMM, no normalization), so
both the CPU oracle and the CUDA path may take their inputs from it.

The shapes and distributions stand in for the production recommendation-model
layers of "LoKA: Low-precision Kernel Applications for Recommendation Models at
Scale" (section II-C, which measures linear layers under learned, heavy-tailed
activation distributions that are not available here):

  * ``single``   X[256,128] ~ N(0,1), W[128,128] ~ N(0,1/128), no bias,
                 per-tensor scaling, LayerNorm (gamma 1, beta 0).
  * ``rec_mlp``  X[65536,512] ~ N(0,1) with 1% of entries multiplied by 100,
                 W[256,512] ~ N(0,1/512), bias ~ N(0,0.02) (variance), per-row
                 scaling, LayerNorm over N=256.
  * ``ensemble`` 8 independent X[32768,256] ~ N(0,1), W[256,256] ~ N(0,1/256),
                 per-row scaling, RMSNorm (eps 1e-6, gamma ~ U(0.5,1.5)).
  * ``mxfp8``    X[262144,2048] ~ Laplace(0,1), W[512,2048] ~ N(0,1/2048),
                 1x32 block scaling with E8M0 scales, LayerNorm over N=512.

Every tensor is returned as a CPU ``torch.bfloat16`` tensor (round-to-nearest
-even from the float32 draw, done by torch's own conversion).  Variances are
written N(mean, variance); "1% of entries" is an independent Bernoulli(0.01)
mask per entry; Laplace(0,1) has scale 1.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

# Variant and normalization identifiers shared by tests and the bench.  These
# are names, not arithmetic.
SCALE_TENSOR, SCALE_ROW, SCALE_MX32, SCALE_BF16, SCALE_BLOCK32 = 0, 1, 2, 3, 4
NORM_NONE, NORM_LAYER, NORM_RMS, NORM_BLOCK_RMS = 0, 1, 2, 3
ACT_NONE, ACT_HARDSWISH = 0, 1
EPS_LAYER = 1e-5
EPS_RMS = 1e-6


@dataclasses.dataclass
class LayerInputs:
    """One linear+norm problem: bf16 tensors on the CPU plus its recipe."""

    x: torch.Tensor                 # [M, K] bf16
    w: torch.Tensor                 # [N, K] bf16 (nn.Linear layout)
    bias: Optional[torch.Tensor]    # [N] bf16 or None
    gamma: Optional[torch.Tensor]   # [N] bf16 or None (=1)
    beta: Optional[torch.Tensor]    # [N] bf16 or None (=0)
    mode: int
    norm: int
    eps: float
    norm_block: int = 256           # NORM_BLOCK_RMS: columns per block
    act: int = ACT_NONE             # activation after the norm

    @property
    def M(self) -> int:
        return self.x.shape[0]

    @property
    def K(self) -> int:
        return self.x.shape[1]

    @property
    def N(self) -> int:
        return self.w.shape[0]


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal(rng: np.random.Generator, shape, var: float = 1.0) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(np.sqrt(var))


def laplace(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    # inverse CDF of Laplace(0, b) from one uniform on (-1/2, 1/2)
    u = rng.random(shape, dtype=np.float32) - np.float32(0.5)
    u = np.clip(u, np.float32(-0.49999997), np.float32(0.49999997))
    return (-np.sign(u) * np.log1p(-2.0 * np.abs(u)) * np.float32(scale)).astype(np.float32)


def with_outliers(rng: np.random.Generator, a: np.ndarray, frac: float, factor: float = 100.0) -> np.ndarray:
    if frac <= 0.0:
        return a
    mask = rng.random(a.shape, dtype=np.float32) < np.float32(frac)
    a = a.copy()
    a[mask] *= np.float32(factor)
    return a


def make_layer(M: int, K: int, N: int, *, mode: int, norm: int, seed: int = 0,
               x_dist: str = "normal", outlier_frac: float = 0.0,
               bias_var: Optional[float] = None, gamma_uniform: bool = False,
               eps: Optional[float] = None) -> LayerInputs:
    """Draw one problem.  The draw order (X, W, bias, gamma) is fixed."""
    rng = np.random.default_rng(seed)
    if x_dist == "normal":
        x = normal(rng, (M, K))
    elif x_dist == "laplace":
        x = laplace(rng, (M, K))
    else:
        raise ValueError(x_dist)
    x = with_outliers(rng, x, outlier_frac)
    w = normal(rng, (N, K), var=1.0 / K)
    bias = _bf16(normal(rng, (N,), var=bias_var)) if bias_var is not None else None
    gamma = _bf16(rng.uniform(0.5, 1.5, size=(N,)).astype(np.float32)) if gamma_uniform else None
    if eps is None:
        eps = EPS_RMS if norm in (NORM_RMS, NORM_BLOCK_RMS) else EPS_LAYER
    return LayerInputs(x=_bf16(x), w=_bf16(w), bias=bias, gamma=gamma, beta=None,
                       mode=mode, norm=norm, eps=eps)


def single(seed: int = 0) -> LayerInputs:
    """Single FP8 linear+LayerNorm, 256x128x128, per-tensor scaling."""
    return make_layer(256, 128, 128, mode=SCALE_TENSOR, norm=NORM_LAYER, seed=seed)


def rec_mlp(seed: int = 0, M: int = 65536, K: int = 512, N: int = 256, mode: int = SCALE_ROW) -> LayerInputs:
    """Recommendation MLP layer with heavy-tailed outliers, per-row scaling
    (or another scaling mode on the same draw)."""
    return make_layer(M, K, N, mode=mode, norm=NORM_LAYER, seed=seed,
                      outlier_frac=0.01, bias_var=0.02)


def ensemble(seed: int = 0, groups: int = 8, M: int = 32768, K: int = 256, N: int = 256) -> List[LayerInputs]:
    """Wide ensemble: independent small GEMMs each followed by RMSNorm."""
    return [make_layer(M, K, N, mode=SCALE_ROW, norm=NORM_RMS, seed=seed * 1000 + g,
                       gamma_uniform=True, eps=EPS_RMS) for g in range(groups)]


def mxfp8(seed: int = 0, M: int = 262144, K: int = 2048, N: int = 512) -> LayerInputs:
    """MXFP8 layer: Laplace activations, 1x32 E8M0 block scaling, LayerNorm."""
    return make_layer(M, K, N, mode=SCALE_MX32, norm=NORM_LAYER, seed=seed, x_dist="laplace")


def wide_blocknorm(seed: int = 0, M: int = 65536, K: int = 512, N: int = 2048) -> LayerInputs:
    """A wide LRM layer: per-row E4M3, BlockNorm over 256-column blocks,
    then Hard Swish (the LoKA Mods pair that keeps wide rows in one pass)."""
    inp = make_layer(M, K, N, mode=SCALE_ROW, norm=NORM_BLOCK_RMS, seed=seed, outlier_frac=0.01, bias_var=0.02)
    inp.norm_block = 256
    inp.act = ACT_HARDSWISH
    return inp


def sweep_shapes():
    """The sweep grid: M in 4096..524288 (powers of two), K, N in 64..2048."""
    Ms = [4096 << i for i in range(8)]
    KN = [64, 128, 256, 512, 1024, 2048]
    return Ms, KN, KN


def random_bf16(shape, seed: int, dist: str = "normal", var: float = 1.0,
                outlier_frac: float = 0.0) -> torch.Tensor:
    """A free-standing seeded bf16 tensor (for quantizer and edge-case tests)."""
    rng = np.random.default_rng(seed)
    a = normal(rng, shape, var) if dist == "normal" else laplace(rng, shape)
    return _bf16(with_outliers(rng, a, outlier_frac))


def all_bf16_patterns() -> torch.Tensor:
    """Every one of the 65,536 bf16 bit patterns, in code order."""
    return torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
