"""GB300-native FP8 linear + normalization for recommendation models.

The compute path is the CUDA library ``libloka.so`` (C ABI in
``include/loka.h``; ctypes binding in ``_loka``).  The helpers below only
allocate device memory with torch and marshal tensors into the C calls:

  quantize_fp8(x, mode)                       -> (q, scales)
  fp8_linear_norm(layers)                     -> [y, ...]   (grouped launch)
  quant_error(x, w, bias, mode)               -> dict of error statistics
  dispatch_select(table, problem, policy)     -> variant id

Sources: "LoKA: Low-precision Kernel Applications for Recommendation Models
at Scale" (sections II-C, III-A, III-B, III-C) and the MXFP8 scaling of the
GEM Training page ("Low Precision Flash Attention").
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

from . import _loka
from ._loka import (LOKA_ACT_HARDSWISH, LOKA_ACT_NONE, LOKA_BF16, LOKA_NORM_BLOCK_RMS,  # noqa: F401
                    LOKA_NORM_LAYER, LOKA_NORM_NONE, LOKA_NORM_RMS, LOKA_SCALE_BLOCK32, LOKA_SCALE_MX32,
                    LOKA_SCALE_ROW, LOKA_SCALE_TENSOR, DispatchEntry, LinearDesc, LokaError, Policy, Problem)

__all__ = ["quantize_fp8", "fp8_linear_norm", "quant_error", "dispatch_select", "Layer", "Workspace"]


def _torch():
    import torch
    return torch


def scales_shape(rows: int, cols: int, mode: int):
    if mode == LOKA_SCALE_TENSOR:
        return (1,), "float32"
    if mode == LOKA_SCALE_ROW:
        return (rows,), "float32"
    if mode == LOKA_SCALE_MX32:
        return (rows, cols // 32), "uint8"
    if mode == LOKA_SCALE_BLOCK32:
        return ((rows + 31) // 32, cols // 32), "uint8"
    raise ValueError(f"mode {mode} has no FP8 scales")


class Workspace:
    """A growable device byte buffer handed to calls that need scratch space."""

    def __init__(self, device=None):
        self.buf = None
        self.device = device

    def get(self, nbytes: int):
        torch = _torch()
        if nbytes == 0:
            return None, 0
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device or "cuda")
        return self.buf, self.buf.numel()


_default_ws = {}


def _ws(device) -> Workspace:
    key = str(device)
    if key not in _default_ws:
        _default_ws[key] = Workspace(device)
    return _default_ws[key]


def quantize_fp8(x, mode: int, workspace: Optional[Workspace] = None, stream=None):
    """E4M3 cast of a bf16 CUDA tensor [rows, cols] whose rows may be strided
    (a column slice of a wider tensor); returns dense (q uint8, scales)."""
    torch = _torch()
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    shp, dt = scales_shape(rows, cols, mode)
    scales = torch.empty(shp, dtype=getattr(torch, dt), device=x.device)
    need = _loka.loka_quantize_fp8_workspace_size(rows, cols, mode)
    ws, nbytes = (workspace or _ws(x.device)).get(need)
    _loka.loka_quantize_fp8(x, rows, cols, x.stride(0), mode, q, scales, ws, nbytes, stream)
    return q, scales


def quantize_fp8_block32(x, transposed: bool = False, stream=None):
    """Square 32x32-block E4M3 cast of a bf16 CUDA tensor [rows, cols];
    returns (q, scales [ceil(rows/32), cols/32], q_t [cols, rows] or None)."""
    torch = _torch()
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous() and x.dim() == 2
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    shp, _ = scales_shape(rows, cols, LOKA_SCALE_BLOCK32)
    scales = torch.empty(shp, dtype=torch.uint8, device=x.device)
    q_t = torch.empty((cols, rows), dtype=torch.uint8, device=x.device) if transposed else None
    _loka.loka_quantize_fp8_block32(x, rows, cols, cols, q, q_t, scales, stream)
    return q, scales, q_t


@dataclasses.dataclass
class Layer:
    """One FP8 linear + norm problem (CUDA tensors)."""

    x: object                      # bf16 [M,K] or uint8 E4M3 [M,K]
    w: object                      # bf16 [N,K] or uint8 E4M3 [N,K]
    mode: int
    norm: int
    eps: float
    bias: object = None
    gamma: object = None
    beta: object = None
    x_scales: object = None        # when x is E4M3
    w_scales: object = None        # when w is E4M3
    y: object = None               # bf16 [M,N] output (allocated if None, unless y_q_only)
    # E4M3 output for the next layer (LOKA_SCALE_ROW or LOKA_SCALE_MX32), or None
    y_q_mode: Optional[int] = None
    y_q: object = None             # uint8 E4M3 [M,N] (allocated if None)
    y_q_scales: object = None      # fp32 [M] or uint8 E8M0 [M,N/32] (allocated if None)
    y_q_only: bool = False         # with y_q_mode: no bf16 copy of the output
    norm_block: int = 256          # LOKA_NORM_BLOCK_RMS: columns per block
    act: int = 0                   # LOKA_ACT_NONE or LOKA_ACT_HARDSWISH

    def desc(self) -> LinearDesc:
        torch = _torch()
        M, K = self.x.shape
        N = self.w.shape[0]
        dev = self.x.device
        quantized_out = self.y_q_mode is not None
        if self.y is None and not (quantized_out and self.y_q_only):
            self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        d = LinearDesc()
        d.M, d.N, d.K = M, N, K
        d.mode, d.norm, d.eps = self.mode, self.norm, self.eps
        d.norm_block, d.act = self.norm_block, self.act
        d.x_is_fp8 = int(self.x.dtype == torch.uint8)
        d.w_is_fp8 = int(self.w.dtype == torch.uint8)
        d.x, d.w = self.x.data_ptr(), self.w.data_ptr()
        d.y = self.y.data_ptr() if self.y is not None else None
        if quantized_out:
            if self.y_q is None:
                self.y_q = torch.empty((M, N), dtype=torch.uint8, device=dev)
            if self.y_q_scales is None:
                shp, dt = scales_shape(M, N, self.y_q_mode)
                self.y_q_scales = torch.empty(shp, dtype=getattr(torch, dt), device=dev)
            d.y_q_mode = self.y_q_mode
            d.y_q, d.y_q_scales = self.y_q.data_ptr(), self.y_q_scales.data_ptr()
        d.x_scales = self.x_scales.data_ptr() if self.x_scales is not None else None
        d.w_scales = self.w_scales.data_ptr() if self.w_scales is not None else None
        d.bias = self.bias.data_ptr() if self.bias is not None else None
        d.gamma = self.gamma.data_ptr() if self.gamma is not None else None
        d.beta = self.beta.data_ptr() if self.beta is not None else None
        return d


def fp8_linear_norm(layers: Sequence[Layer], workspace: Optional[Workspace] = None, stream=None) -> List[object]:
    """Runs all layers in one grouped call; returns their bf16 outputs."""
    descs = [l.desc() for l in layers]
    need = _loka.loka_fp8_linear_norm_workspace_size(descs)
    ws, nbytes = (workspace or _ws(layers[0].x.device)).get(need)
    _loka.loka_fp8_linear_norm(descs, ws, nbytes, stream)
    return [l.y for l in layers]


def quant_error(x, w, bias, mode: int, norm: int = LOKA_NORM_NONE, eps: float = 0.0, gamma=None, beta=None,
                norm_block: int = 256, act: int = LOKA_ACT_NONE, workspace: Optional[Workspace] = None,
                stream=None) -> dict:
    """Probe: FP8 (mode) vs high-precision outputs of one layer, before and
    after its normalization."""
    layer = Layer(x=x, w=w, bias=bias, gamma=gamma, beta=beta, mode=mode, norm=norm, eps=eps,
                  norm_block=norm_block, act=act, y=x.new_empty((0,)))
    d = layer.desc()
    d.y = None
    need = _loka.loka_quant_error_workspace_size(d)
    ws, nbytes = (workspace or _ws(x.device)).get(need)
    st = _loka.loka_quant_error(d, ws, nbytes, stream)
    return {"mere": st.mere, "rel_err_fro": st.rel_err_fro, "max_abs": st.max_abs,
            "max_abs_post_norm": st.max_abs_post_norm, "zero_ref_count": st.zero_ref_count, "count": st.count}


class InputStats:
    """LoKA Probe's running input statistics of one layer (count, fp64 mean
    and scatter matrix on the device), updated batch by batch on the GPU."""

    def __init__(self, K: int, device):
        torch = _torch()
        self.device = torch.device(device)
        self.mu = torch.zeros(K, dtype=torch.float64, device=self.device)
        self.scatter = torch.zeros((K, K), dtype=torch.float64, device=self.device)
        self.c = _loka.InputStats()
        self.c.n, self.c.K = 0, K
        self.c.mu, self.c.scatter = self.mu.data_ptr(), self.scatter.data_ptr()

    @property
    def n(self) -> int:
        return self.c.n

    def update(self, x, workspace: Optional[Workspace] = None, stream=None) -> None:
        """Merge the rows of x (bf16 CUDA [B, K])."""
        B = x.shape[0]
        need = _loka.loka_probe_stats_workspace_size(B, self.c.K)
        ws, nbytes = (workspace or _ws(self.device)).get(need)
        _loka.loka_probe_stats_update(self.c, x, B, ws, nbytes, stream)

    def covariance(self, stream=None):
        """The unbiased covariance scatter / (n - 1), computed by the library
        into a new fp64 CUDA tensor [K, K]."""
        torch = _torch()
        K = self.c.K
        cov = torch.empty((K, K), dtype=torch.float64, device=self.device)
        _loka.loka_probe_covariance(self.c, cov, stream)
        return cov

    def factor(self, eps_rel: float = 1e-6, workspace: Optional[Workspace] = None, stream=None):
        """(L, mu) in bf16 for sample_inputs: L L^T = covariance + eps I."""
        torch = _torch()
        K = self.c.K
        L = torch.empty((K, K), dtype=torch.bfloat16, device=self.device)
        mu = torch.empty(K, dtype=torch.bfloat16, device=self.device)
        need = _loka.loka_probe_cholesky_workspace_size(K)
        ws, nbytes = (workspace or _ws(self.device)).get(need)
        _loka.loka_probe_cholesky(self.c, eps_rel, L, mu, ws, nbytes, stream)
        return L, mu


class WeightModel:
    """LoKA Probe's matrix-normal model of one weight [R, C]: fp32 mean,
    row covariance U and column covariance V on the device, updated weight by
    weight on the GPU (loka_probe_weight_update)."""

    def __init__(self, R: int, C: int, device):
        torch = _torch()
        self.device = torch.device(device)
        self.mean = torch.zeros((R, C), dtype=torch.float32, device=self.device)
        self.U = torch.zeros((R, R), dtype=torch.float32, device=self.device)
        self.V = torch.zeros((C, C), dtype=torch.float32, device=self.device)
        self.c = _loka.WeightStats()
        self.c.n, self.c.R, self.c.C = 0, R, C
        self.c.mean, self.c.U, self.c.V = self.mean.data_ptr(), self.U.data_ptr(), self.V.data_ptr()

    @property
    def n(self) -> int:
        return self.c.n

    def _ws(self, workspace):
        need = _loka.loka_probe_weight_workspace_size(self.c.R, self.c.C)
        return (workspace or _ws(self.device)).get(need)

    def update(self, w, momentum: float = 0.95, eps_rel: float = 1e-6, workspace: Optional[Workspace] = None,
               stream=None) -> None:
        """Merge the weight w (bf16 CUDA [R, C])."""
        ws, nbytes = self._ws(workspace)
        _loka.loka_probe_weight_update(self.c, w, momentum, eps_rel, ws, nbytes, stream)

    def sample(self, seed: int, eps_rel: float = 1e-6, workspace: Optional[Workspace] = None, stream=None):
        """A synthetic weight M + L_U Z L_V^T (bf16 CUDA [R, C])."""
        torch = _torch()
        out = torch.empty((self.c.R, self.c.C), dtype=torch.bfloat16, device=self.device)
        ws, nbytes = self._ws(workspace)
        _loka.loka_probe_sample_weights(self.c, eps_rel, seed, out, ws, nbytes, stream)
        return out


def sample_inputs(mu, chol, B: int, seed: int, workspace: Optional[Workspace] = None, stream=None):
    """B synthetic input rows Z L^T + mu (bf16 CUDA [B, K]); mu bf16 [K], chol
    the bf16 [K, K] lower Cholesky factor of the regularized covariance."""
    torch = _torch()
    K = mu.shape[0]
    out = torch.empty((B, K), dtype=torch.bfloat16, device=mu.device)
    need = _loka.loka_probe_sample_workspace_size(B, K)
    ws, nbytes = (workspace or _ws(mu.device)).get(need)
    _loka.loka_probe_sample_inputs(mu, chol, B, K, seed, out, ws, nbytes, stream)
    return out


def dispatch_select(table, M: int, N: int, K: int, norm: int, outlier_frac: float,
                    max_rel_err: float = 1e-2, max_mere: float = 0.2, min_speedup: float = -1.0) -> int:
    """table: iterable of (M, N, K, norm, outlier_frac, variant, time_us, rel_err, mere)."""
    rows = []
    for (m, n, k, nm, o, v, t, r, me) in table:
        e = DispatchEntry()
        e.p.M, e.p.N, e.p.K, e.p.norm, e.p.outlier_frac = m, n, k, nm, o
        e.variant, e.time_us, e.rel_err, e.mere = v, t, r, me
        rows.append(e)
    p = Problem()
    p.M, p.N, p.K, p.norm, p.outlier_frac = M, N, K, norm, outlier_frac
    pol = Policy()
    pol.max_rel_err, pol.max_mere, pol.min_speedup = max_rel_err, max_mere, min_speedup
    return _loka.loka_dispatch_select(rows, p, pol)
