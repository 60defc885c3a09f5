"""ctypes binding of the C ABI in include/loka.h.

Argument marshalling only: every function here converts Python/torch
arguments to the plain pointers and sizes of the C call and calls it.  The
computation runs in the library's CUDA kernels; there is no Python or CPU
fallback, and loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libloka.so")

LOKA_OK, LOKA_ERR_INVALID_ARG, LOKA_ERR_UNSUPPORTED, LOKA_ERR_WORKSPACE, LOKA_ERR_TIMEOUT, LOKA_ERR_CUDA, \
    LOKA_ERR_NUMERIC = range(7)
LOKA_SCALE_TENSOR, LOKA_SCALE_ROW, LOKA_SCALE_MX32, LOKA_BF16, LOKA_SCALE_BLOCK32 = range(5)
LOKA_NORM_NONE, LOKA_NORM_LAYER, LOKA_NORM_RMS, LOKA_NORM_BLOCK_RMS = range(4)
LOKA_ACT_NONE, LOKA_ACT_HARDSWISH = range(2)

c_i64, c_i32, c_sz, c_p = ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p


class LinearDesc(ctypes.Structure):
    _fields_ = [("M", c_i64), ("N", c_i64), ("K", c_i64), ("mode", c_i32), ("norm", c_i32),
                ("eps", ctypes.c_float), ("x_is_fp8", c_i32), ("w_is_fp8", c_i32), ("y_q_mode", c_i32),
                ("x", c_p), ("x_scales", c_p), ("w", c_p), ("w_scales", c_p), ("bias", c_p),
                ("gamma", c_p), ("beta", c_p), ("y", c_p), ("y_q", c_p), ("y_q_scales", c_p),
                ("norm_block", c_i32), ("act", c_i32)]


class ErrorStats(ctypes.Structure):
    _fields_ = [("mere", ctypes.c_double), ("rel_err_fro", ctypes.c_double), ("max_abs", ctypes.c_double),
                ("max_abs_post_norm", ctypes.c_double), ("zero_ref_count", c_i64), ("count", c_i64)]


class Problem(ctypes.Structure):
    _fields_ = [("M", c_i64), ("N", c_i64), ("K", c_i64), ("norm", c_i32), ("reserved", c_i32),
                ("outlier_frac", ctypes.c_double)]


class DispatchEntry(ctypes.Structure):
    _fields_ = [("p", Problem), ("variant", c_i32), ("reserved", c_i32), ("time_us", ctypes.c_double),
                ("rel_err", ctypes.c_double), ("mere", ctypes.c_double)]


class InputStats(ctypes.Structure):
    _fields_ = [("n", c_i64), ("K", c_i64), ("mu", c_p), ("scatter", c_p)]


class WeightStats(ctypes.Structure):
    _fields_ = [("n", c_i64), ("R", c_i64), ("C", c_i64), ("mean", c_p), ("U", c_p), ("V", c_p)]


class Policy(ctypes.Structure):
    _fields_ = [("max_rel_err", ctypes.c_double), ("max_mere", ctypes.c_double), ("min_speedup", ctypes.c_double)]


# name -> (restype, argtypes)
SIGNATURES = {
    "loka_version": (c_i32, []),
    "loka_last_error": (ctypes.c_char_p, []),
    "loka_device_status": (c_i32, [c_p]),
    "loka_selftest_watchdog": (c_i32, [ctypes.c_uint64, c_p]),
    "loka_selftest_mma_peak": (c_i32, [c_i32, ctypes.c_int64, c_p]),
    "loka_quantize_fp8_workspace_size": (c_sz, [c_i64, c_i64, c_i32]),
    "loka_quantize_fp8": (c_i32, [c_p, c_i64, c_i64, c_i64, c_i32, c_p, c_p, c_p, c_sz, c_p]),
    "loka_quantize_fp8_block32": (c_i32, [c_p, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p]),
    "loka_probe_stats_workspace_size": (c_sz, [c_i64, c_i64]),
    "loka_probe_stats_update": (c_i32, [ctypes.POINTER(InputStats), c_p, c_i64, c_p, c_sz, c_p]),
    "loka_probe_sample_workspace_size": (c_sz, [c_i64, c_i64]),
    "loka_probe_covariance": (c_i32, [ctypes.POINTER(InputStats), c_p, c_p]),
    "loka_probe_cholesky_workspace_size": (c_sz, [c_i64]),
    "loka_probe_cholesky": (c_i32, [ctypes.POINTER(InputStats), ctypes.c_double, c_p, c_p, c_p, c_sz, c_p]),
    "loka_probe_sample_inputs": (c_i32, [c_p, c_p, c_i64, c_i64, ctypes.c_uint64, c_p, c_p, c_sz, c_p]),
    "loka_probe_weight_workspace_size": (c_sz, [c_i64, c_i64]),
    "loka_probe_weight_update": (c_i32, [ctypes.POINTER(WeightStats), c_p, ctypes.c_double, ctypes.c_double, c_p,
                                         c_sz, c_p]),
    "loka_probe_sample_weights": (c_i32, [ctypes.POINTER(WeightStats), ctypes.c_double, ctypes.c_uint64, c_p, c_p,
                                          c_sz, c_p]),
    "loka_fp8_linear_norm_workspace_size": (c_sz, [ctypes.POINTER(LinearDesc), c_i32]),
    "loka_fp8_linear_norm": (c_i32, [ctypes.POINTER(LinearDesc), c_i32, c_p, c_sz, c_p]),
    "loka_fp8_linear_norm_static": (c_i32, [ctypes.POINTER(LinearDesc), c_i32, c_p]),
    "loka_quant_error_workspace_size": (c_sz, [ctypes.POINTER(LinearDesc)]),
    "loka_quant_error": (c_i32, [ctypes.POINTER(LinearDesc), c_p, c_sz, ctypes.POINTER(ErrorStats), c_p]),
    "loka_dispatch_select": (c_i32, [ctypes.POINTER(DispatchEntry), c_i64, ctypes.POINTER(Problem),
                                     ctypes.POINTER(Policy), ctypes.POINTER(c_i32)]),
}

_lib = None
_lock = threading.Lock()


class LokaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"loka status {status}: {message}")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the library once; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                                   "(there is no CPU fallback)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def check(status: int) -> None:
    if status != LOKA_OK:
        msg = load().loka_last_error()
        raise LokaError(status, msg.decode() if msg else "")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------- same-name calls
def loka_version() -> int:
    return load().loka_version()


def loka_device_status(stream=None) -> int:
    return load().loka_device_status(_stream(stream))


def loka_selftest_watchdog(limit_ns: int, stream=None) -> None:
    check(load().loka_selftest_watchdog(limit_ns, _stream(stream)))


def loka_selftest_mma_peak(kind: int, mmas_per_sm: int, stream=None) -> None:
    check(load().loka_selftest_mma_peak(kind, mmas_per_sm, _stream(stream)))


def loka_quantize_fp8_workspace_size(rows: int, cols: int, mode: int) -> int:
    return load().loka_quantize_fp8_workspace_size(rows, cols, mode)


def loka_quantize_fp8(x, rows: int, cols: int, ld: int, mode: int, q, scales, workspace=None,
                      workspace_bytes: int = 0, stream=None) -> None:
    check(load().loka_quantize_fp8(_ptr(x), rows, cols, ld, mode, _ptr(q), _ptr(scales), _ptr(workspace),
                                   workspace_bytes, _stream(stream)))


def loka_quantize_fp8_block32(x, rows: int, cols: int, ld: int, q, q_t, scales, stream=None) -> None:
    check(load().loka_quantize_fp8_block32(_ptr(x), rows, cols, ld, _ptr(q), _ptr(q_t), _ptr(scales),
                                           _stream(stream)))


def loka_probe_stats_workspace_size(B: int, K: int) -> int:
    return load().loka_probe_stats_workspace_size(B, K)


def loka_probe_stats_update(stats: InputStats, x, B: int, workspace, workspace_bytes: int, stream=None) -> None:
    check(load().loka_probe_stats_update(ctypes.byref(stats), _ptr(x), B, _ptr(workspace), workspace_bytes,
                                         _stream(stream)))


def loka_probe_covariance(stats: InputStats, cov, stream=None) -> None:
    check(load().loka_probe_covariance(ctypes.byref(stats), _ptr(cov), _stream(stream)))


def loka_probe_cholesky_workspace_size(K: int) -> int:
    return load().loka_probe_cholesky_workspace_size(K)


def loka_probe_cholesky(stats: InputStats, eps_rel: float, chol, mu_out, workspace, workspace_bytes: int,
                        stream=None) -> None:
    check(load().loka_probe_cholesky(ctypes.byref(stats), eps_rel, _ptr(chol), _ptr(mu_out), _ptr(workspace),
                                     workspace_bytes, _stream(stream)))


def loka_probe_sample_workspace_size(B: int, K: int) -> int:
    return load().loka_probe_sample_workspace_size(B, K)


def loka_probe_sample_inputs(mu, chol, B: int, K: int, seed: int, out, workspace, workspace_bytes: int,
                             stream=None) -> None:
    check(load().loka_probe_sample_inputs(_ptr(mu), _ptr(chol), B, K, seed, _ptr(out), _ptr(workspace),
                                          workspace_bytes, _stream(stream)))


def loka_probe_weight_workspace_size(R: int, C: int) -> int:
    return load().loka_probe_weight_workspace_size(R, C)


def loka_probe_weight_update(stats: WeightStats, w, momentum: float, eps_rel: float, workspace, workspace_bytes: int,
                             stream=None) -> None:
    check(load().loka_probe_weight_update(ctypes.byref(stats), _ptr(w), momentum, eps_rel, _ptr(workspace),
                                          workspace_bytes, _stream(stream)))


def loka_probe_sample_weights(stats: WeightStats, eps_rel: float, seed: int, out, workspace, workspace_bytes: int,
                              stream=None) -> None:
    check(load().loka_probe_sample_weights(ctypes.byref(stats), eps_rel, seed, _ptr(out), _ptr(workspace),
                                           workspace_bytes, _stream(stream)))


def make_descs(descs: Sequence[LinearDesc]):
    arr = (LinearDesc * len(descs))(*descs)
    return arr


def loka_fp8_linear_norm_workspace_size(descs: Sequence[LinearDesc]) -> int:
    arr = make_descs(descs)
    return load().loka_fp8_linear_norm_workspace_size(arr, len(descs))


def loka_fp8_linear_norm(descs: Sequence[LinearDesc], workspace=None, workspace_bytes: int = 0, stream=None) -> None:
    arr = make_descs(descs)
    check(load().loka_fp8_linear_norm(arr, len(descs), _ptr(workspace), workspace_bytes, _stream(stream)))


def loka_fp8_linear_norm_static(descs: Sequence[LinearDesc], stream=None) -> None:
    """loka_fp8_linear_norm with the library's built-in scratch (no workspace,
    no allocation; for callers that cannot allocate device memory)."""
    arr = make_descs(descs)
    check(load().loka_fp8_linear_norm_static(arr, len(descs), _stream(stream)))


def loka_quant_error_workspace_size(desc: LinearDesc) -> int:
    return load().loka_quant_error_workspace_size(ctypes.byref(desc))


def loka_quant_error(desc: LinearDesc, workspace, workspace_bytes: int, stream=None) -> ErrorStats:
    st = ErrorStats()
    check(load().loka_quant_error(ctypes.byref(desc), _ptr(workspace), workspace_bytes, ctypes.byref(st),
                                  _stream(stream)))
    return st


def loka_dispatch_select(table: Sequence[DispatchEntry], problem: Problem, policy: Policy) -> int:
    arr = (DispatchEntry * max(1, len(table)))(*table)
    out = c_i32(-1)
    check(load().loka_dispatch_select(arr, len(table), ctypes.byref(problem), ctypes.byref(policy),
                                      ctypes.byref(out)))
    return out.value
