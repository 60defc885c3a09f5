"""CPU checks of the C-ABI library: it builds, loads, exports every symbol the
header declares, rejects bad arguments on the host before any launch, and its
host-only dispatch selector agrees with the oracle's reading of the rule."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import dispatch as D
from fp8_precision_recommendation_gb300 import _loka

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "loka.h")


@pytest.fixture(scope="module")
def cpu_lib():
    if not os.path.exists(_loka.LIB_PATH):
        from fp8_precision_recommendation_gb300 import build
        build.build()
    return _loka.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(loka_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ["loka_quantize_fp8", "loka_fp8_linear_norm", "loka_quant_error", "loka_dispatch_select"]:
        assert n in names


def test_library_exports_every_declared_symbol(cpu_lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(cpu_lib, n), n
        assert n in _loka.SIGNATURES, n


def test_struct_layouts_match_header(tmp_path):
    # the C compiler's sizeof / offsetof of every struct and field of the
    # header against the ctypes binding
    structs = {"loka_linear_desc": _loka.LinearDesc, "loka_error_stats": _loka.ErrorStats,
               "loka_problem": _loka.Problem, "loka_dispatch_entry": _loka.DispatchEntry,
               "loka_policy": _loka.Policy, "loka_input_stats": _loka.InputStats,
               "loka_weight_stats": _loka.WeightStats}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "loka.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, cls in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert got[(cname, fname)] == getattr(cls, fname).offset, (cname, fname)


def test_version(cpu_lib):
    assert _loka.loka_version() >= 1


def _desc(**kw):
    d = _loka.LinearDesc()
    d.M, d.N, d.K, d.mode, d.norm, d.eps = 256, 256, 512, 1, 1, 1e-5
    d.x = d.w = d.y = 1 << 20
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("kw,status", [
    ({"N": 100}, _loka.LOKA_ERR_UNSUPPORTED), ({"N": 4096}, _loka.LOKA_ERR_UNSUPPORTED),
    ({"N": 16}, _loka.LOKA_ERR_UNSUPPORTED), ({"K": 80}, _loka.LOKA_ERR_UNSUPPORTED),
    ({"K": 16}, _loka.LOKA_ERR_UNSUPPORTED),
    # any multiple of 32 passes validation (then the missing workspace stops it)
    ({"K": 96}, _loka.LOKA_ERR_WORKSPACE), ({"K": 32}, _loka.LOKA_ERR_WORKSPACE),
    ({"N": 96}, _loka.LOKA_ERR_WORKSPACE), ({"N": 768}, _loka.LOKA_ERR_WORKSPACE),
    ({"N": 2016, "norm": 2}, _loka.LOKA_ERR_WORKSPACE), ({"N": 320, "mode": 2}, _loka.LOKA_ERR_WORKSPACE),
    ({"M": -1}, _loka.LOKA_ERR_INVALID_ARG),
    ({"mode": 7}, _loka.LOKA_ERR_INVALID_ARG),
    ({"norm": 9}, _loka.LOKA_ERR_INVALID_ARG),
    ({"eps": float("nan")}, _loka.LOKA_ERR_INVALID_ARG),
    ({"x": None}, _loka.LOKA_ERR_INVALID_ARG),
    ({"y": (1 << 20) + 8}, _loka.LOKA_ERR_INVALID_ARG),         # misaligned
    ({"mode": 3, "x_is_fp8": 1, "x_scales": 64}, _loka.LOKA_ERR_INVALID_ARG),
    ({"x_is_fp8": 1}, _loka.LOKA_ERR_INVALID_ARG),                # no x_scales
])
def test_linear_norm_rejects_bad_arguments_on_host(cpu_lib, kw, status):
    arr = _loka.make_descs([_desc(**kw)])
    assert cpu_lib.loka_fp8_linear_norm(arr, 1, None, 0, None) == status
    assert len(cpu_lib.loka_last_error()) > 0


def test_linear_norm_rejects_group_count_and_mismatch(cpu_lib):
    arr = _loka.make_descs([_desc()])
    assert cpu_lib.loka_fp8_linear_norm(arr, 0, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG
    assert cpu_lib.loka_fp8_linear_norm(arr, 17, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG
    arr2 = _loka.make_descs([_desc(), _desc(K=256)])
    assert cpu_lib.loka_fp8_linear_norm(arr2, 2, None, 0, None) == _loka.LOKA_ERR_UNSUPPORTED


_Q = 1 << 21     # a fake 16-byte-aligned device address (nothing is launched)


@pytest.mark.parametrize("kw,status", [
    ({"y_q_mode": 0}, _loka.LOKA_ERR_UNSUPPORTED),                  # a tensor-wide output scale
    ({"y_q_mode": 5}, _loka.LOKA_ERR_INVALID_ARG),
    ({"y_q_mode": 1, "N": 512}, _loka.LOKA_ERR_UNSUPPORTED),        # a row scale across a cluster
    ({"y_q_mode": 1, "mode": 3}, _loka.LOKA_ERR_UNSUPPORTED),       # the bf16 path
    ({"y_q_mode": 1, "y_q_scales": None}, _loka.LOKA_ERR_INVALID_ARG),
    ({"y_q_mode": 1, "y_q": _Q + 8}, _loka.LOKA_ERR_INVALID_ARG),   # misaligned codes
    ({"y_q_mode": 1, "y_q_scales": _Q + 2}, _loka.LOKA_ERR_INVALID_ARG),
    ({"y_q_mode": 1, "y": None}, _loka.LOKA_ERR_WORKSPACE),         # valid: the bf16 copy is optional
    ({"y_q_mode": 2, "N": 2048, "y_q_scales": _Q + 1}, _loka.LOKA_ERR_WORKSPACE),   # MX: any N, byte scales
    ({"y_q_mode": 1, "mode": 0}, _loka.LOKA_ERR_WORKSPACE),         # per-tensor inputs, per-row output
])
def test_quantized_output_arguments_on_host(cpu_lib, kw, status):
    kw = dict({"y_q": _Q, "y_q_scales": _Q}, **kw)
    arr = _loka.make_descs([_desc(**kw)])
    assert cpu_lib.loka_fp8_linear_norm(arr, 1, None, 0, None) == status, cpu_lib.loka_last_error()


@pytest.mark.parametrize("kw,status", [
    ({"norm": 3, "norm_block": 48}, _loka.LOKA_ERR_UNSUPPORTED),       # blocks are 32..256, powers of two
    ({"norm": 3, "norm_block": 512}, _loka.LOKA_ERR_UNSUPPORTED),
    ({"norm": 3, "norm_block": 128, "N": 192}, _loka.LOKA_ERR_INVALID_ARG),   # does not divide N
    ({"norm": 4}, _loka.LOKA_ERR_INVALID_ARG),
    ({"act": 2}, _loka.LOKA_ERR_INVALID_ARG),
    ({"norm": 3, "norm_block": 64, "N": 192, "act": 1}, _loka.LOKA_ERR_WORKSPACE),   # valid
    ({"norm": 3, "norm_block": 256, "N": 2048}, _loka.LOKA_ERR_WORKSPACE),           # valid, wide rows
    ({"norm": 0, "act": 1}, _loka.LOKA_ERR_WORKSPACE),                               # activation alone
])
def test_blocknorm_and_activation_arguments_on_host(cpu_lib, kw, status):
    arr = _loka.make_descs([_desc(**kw)])
    assert cpu_lib.loka_fp8_linear_norm(arr, 1, None, 0, None) == status, cpu_lib.loka_last_error()


def test_groups_share_norm_block_and_activation(cpu_lib):
    a = {"norm": 3, "norm_block": 64}
    assert cpu_lib.loka_fp8_linear_norm(_loka.make_descs([_desc(**a), _desc(norm=3, norm_block=128)]), 2, None, 0,
                                        None) == _loka.LOKA_ERR_UNSUPPORTED
    assert cpu_lib.loka_fp8_linear_norm(_loka.make_descs([_desc(act=1), _desc()]), 2, None, 0, None) == \
        _loka.LOKA_ERR_UNSUPPORTED


def test_quantized_output_is_all_groups_or_none(cpu_lib):
    q = {"y_q": _Q, "y_q_scales": _Q, "y_q_mode": 1}
    assert cpu_lib.loka_fp8_linear_norm(_loka.make_descs([_desc(**q), _desc()]), 2, None, 0, None) == \
        _loka.LOKA_ERR_UNSUPPORTED
    assert cpu_lib.loka_fp8_linear_norm(_loka.make_descs([_desc(**q), _desc(**dict(q, y_q_mode=2))]), 2, None, 0,
                                        None) == _loka.LOKA_ERR_UNSUPPORTED
    assert cpu_lib.loka_fp8_linear_norm(_loka.make_descs([_desc(**q), _desc(**q)]), 2, None, 0, None) == \
        _loka.LOKA_ERR_WORKSPACE
    # an empty group has no output storage: it does not count
    assert cpu_lib.loka_fp8_linear_norm(_loka.make_descs([_desc(M=0, y=None), _desc(**q)]), 2, None, 0, None) == \
        _loka.LOKA_ERR_WORKSPACE
    # without y_q, y stays required
    assert cpu_lib.loka_fp8_linear_norm(_loka.make_descs([_desc(y=None)]), 1, None, 0, None) == \
        _loka.LOKA_ERR_INVALID_ARG


def test_linear_norm_workspace_is_required_and_sized(cpu_lib):
    al = lambda n: (n + 255) // 256 * 256
    # rowwise: X E4M3 + row scales + W E4M3 + row scales, each 256-byte aligned
    d = _desc()
    need = _loka.loka_fp8_linear_norm_workspace_size([d])
    assert need == al(256 * 512) + al(256 * 4) + al(256 * 512) + al(256 * 4)
    # tensorwise: X and W codes, scales and the two amax slots
    need3 = _loka.loka_fp8_linear_norm_workspace_size([_desc(mode=0)])
    assert need3 == 2 * al(256 * 512) + 2 * al(4) + al(8)
    arr = _loka.make_descs([d])
    assert cpu_lib.loka_fp8_linear_norm(arr, 1, None, 0, None) == _loka.LOKA_ERR_WORKSPACE
    assert _loka.loka_fp8_linear_norm_workspace_size([_desc(mode=3)]) == 0


def test_quantize_rejects_bad_arguments_on_host(cpu_lib):
    f = cpu_lib.loka_quantize_fp8
    assert f(1 << 20, 4, 48, 48, 1, 1 << 20, 1 << 20, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG   # cols % 32
    assert f(1 << 20, 4, 64, 64, 5, 1 << 20, 1 << 20, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG   # mode
    assert f(None, 4, 64, 64, 1, 1 << 20, 1 << 20, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG
    assert f((1 << 20) + 2, 4, 64, 64, 1, 1 << 20, 1 << 20, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG
    assert f(1 << 20, 4, 64, 32, 1, 1 << 20, 1 << 20, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG   # ld < cols
    assert f(1 << 20, 4, 64, 68, 1, 1 << 20, 1 << 20, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG   # ld % 8
    assert f(1 << 20, 4, 64, 64, 0, 1 << 20, 1 << 20, None, 0, None) == _loka.LOKA_ERR_WORKSPACE
    assert _loka.loka_quantize_fp8_workspace_size(4, 64, 0) > 0
    assert _loka.loka_quantize_fp8_workspace_size(4, 64, 1) == 0


def test_block32_quantizer_rejects_bad_arguments_on_host(cpu_lib):
    f = cpu_lib.loka_quantize_fp8_block32
    assert f(1 << 20, 48, 64, 64, 1 << 20, 1 << 21, 1 << 22, None) == _loka.LOKA_ERR_INVALID_ARG   # q_t: rows % 32
    assert f(1 << 20, 64, 48, 48, 1 << 20, None, 1 << 22, None) == _loka.LOKA_ERR_INVALID_ARG      # cols % 32
    assert f(1 << 20, 64, 64, 64, (1 << 20) + 8, None, 1 << 22, None) == _loka.LOKA_ERR_INVALID_ARG  # q alignment
    assert f(1 << 20, 64, 64, 64, 1 << 20, (1 << 21) + 8, 1 << 22, None) == _loka.LOKA_ERR_INVALID_ARG
    assert f(1 << 20, 0, 64, 64, 1 << 20, None, 1 << 22, None) == _loka.LOKA_OK                    # empty


def test_probe_statistics_reject_bad_arguments_on_host(cpu_lib):
    st = _loka.InputStats()
    st.n, st.K, st.mu, st.scatter = 0, 64, 1 << 20, 1 << 21
    upd = cpu_lib.loka_probe_stats_update
    assert upd(ctypes.byref(st), 1 << 22, 1000, None, 0, None) == _loka.LOKA_ERR_UNSUPPORTED     # K = 64
    st.K = 512
    assert upd(None, 1 << 22, 1000, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG
    assert upd(ctypes.byref(st), (1 << 22) + 8, 1000, None, 0, None) == _loka.LOKA_ERR_INVALID_ARG   # x alignment
    assert upd(ctypes.byref(st), 1 << 22, 1000, None, 0, None) == _loka.LOKA_ERR_WORKSPACE
    assert upd(ctypes.byref(st), 1 << 22, 0, None, 0, None) == _loka.LOKA_OK and st.n == 0     # empty batch
    # workspace: X^T in split-K groups (zero-padded to 128 rows) + sums + partials
    assert _loka.loka_probe_stats_workspace_size(65536, 512) >= 65536 * 512 * 2 + 16 * 512 * 512 * 4
    smp = cpu_lib.loka_probe_sample_inputs
    assert smp(1 << 20, 1 << 21, 100, 96, 1, 1 << 22, None, 0, None) == _loka.LOKA_ERR_UNSUPPORTED
    assert smp(1 << 20, 1 << 21, 100, 256, 1, 1 << 22, None, 0, None) == _loka.LOKA_ERR_WORKSPACE


def test_probe_covariance_rejects_bad_arguments_on_host(cpu_lib):
    st = _loka.InputStats()
    st.n, st.K, st.mu, st.scatter = 1, 64, 1 << 20, 1 << 21
    cov = cpu_lib.loka_probe_covariance
    assert cov(ctypes.byref(st), 1 << 22, None) == _loka.LOKA_ERR_INVALID_ARG          # n < 2
    st.n = 10
    assert cov(None, 1 << 22, None) == _loka.LOKA_ERR_INVALID_ARG
    assert cov(ctypes.byref(st), None, None) == _loka.LOKA_ERR_INVALID_ARG
    assert cov(ctypes.byref(st), (1 << 22) + 4, None) == _loka.LOKA_ERR_INVALID_ARG    # alignment
    st.scatter = None
    assert cov(ctypes.byref(st), 1 << 22, None) == _loka.LOKA_ERR_INVALID_ARG


def test_weight_model_rejects_bad_arguments_on_host(cpu_lib):
    st = _loka.WeightStats()
    st.n, st.R, st.C, st.mean, st.U, st.V = 0, 64, 96, 1 << 20, 1 << 21, 1 << 22
    upd = cpu_lib.loka_probe_weight_update
    assert upd(ctypes.byref(st), 1 << 23, 0.9, 1e-6, None, 0, None) == _loka.LOKA_ERR_WORKSPACE
    need = _loka.loka_probe_weight_workspace_size(64, 96)
    assert need >= 3 * 64 * 96 * 4 + 2 * 64 * 64 * 4 + 2 * 96 * 96 * 4
    assert upd(ctypes.byref(st), 1 << 23, 1.0, 1e-6, 1 << 24, need, None) == _loka.LOKA_ERR_INVALID_ARG   # momentum
    assert upd(ctypes.byref(st), None, 0.9, 1e-6, 1 << 24, need, None) == _loka.LOKA_ERR_INVALID_ARG
    st.C = 97
    assert upd(ctypes.byref(st), 1 << 23, 0.9, 1e-6, 1 << 24, need, None) == _loka.LOKA_ERR_UNSUPPORTED  # odd C
    st.C, st.R = 96, 4096
    assert upd(ctypes.byref(st), 1 << 23, 0.9, 1e-6, 1 << 24, need, None) == _loka.LOKA_ERR_UNSUPPORTED  # R too large
    assert _loka.loka_probe_weight_workspace_size(4096, 96) == 0
    st.R = 64
    smp = cpu_lib.loka_probe_sample_weights
    assert smp(ctypes.byref(st), 1e-6, 1, 1 << 23, 1 << 24, need, None) == _loka.LOKA_ERR_INVALID_ARG    # n == 0


def _c_table(rows):
    out = []
    for e in rows:
        d = _loka.DispatchEntry()
        d.p.M, d.p.N, d.p.K, d.p.norm, d.p.outlier_frac = e.M, e.N, e.K, e.norm, e.outlier_frac
        d.variant, d.time_us, d.rel_err, d.mere = e.variant, e.time_us, e.rel_err, e.mere
        out.append(d)
    return out


def _c_select(rows, M, N, K, norm, o, pol):
    p = _loka.Problem()
    p.M, p.N, p.K, p.norm, p.outlier_frac = M, N, K, norm, o
    c = _loka.Policy()
    c.max_rel_err, c.max_mere, c.min_speedup = pol.max_rel_err, pol.max_mere, pol.min_speedup
    return _loka.loka_dispatch_select(_c_table(rows), p, c)


def test_dispatch_select_agrees_with_oracle_on_random_tables(cpu_lib):
    rng = np.random.default_rng(3)
    Ms = [4096, 16384, 65536]
    for trial in range(300):
        rows = []
        for m in Ms:
            for o in (0.0, 0.01):
                for v in range(4):
                    if rng.random() < 0.85:
                        rows.append(D.Entry(m, 256, 512, 1, o, v, float(rng.integers(1, 6)),
                                            float(rng.choice([1e-3, 5e-3, 2e-2])), float(rng.choice([0.05, 0.1, 0.3]))))
        pol = D.Policy(max_rel_err=float(rng.choice([1e-2, 1e-1])), max_mere=float(rng.choice([0.2, -1.0])),
                       min_speedup=float(rng.choice([1.05, -1.0])))
        M = int(rng.choice([3000, 8192, 30000, 65536, 100000]))
        o = float(rng.choice([0.0, 0.004, 0.02]))
        assert _c_select(rows, M, 256, 512, 1, o, pol) == D.select(rows, M, 256, 512, 1, o, pol)


def test_dispatch_select_empty_table_is_bf16(cpu_lib):
    p = _loka.Problem()
    p.M, p.N, p.K, p.norm = 1024, 256, 512, 1
    pol = _loka.Policy()
    pol.max_rel_err, pol.max_mere, pol.min_speedup = 1e-2, 0.2, 1.05
    assert _loka.loka_dispatch_select([], p, pol) == _loka.LOKA_BF16


def test_measured_dispatch_table_agrees_with_oracle_selection(cpu_lib):
    # the committed table is the variant sweep measured on a GB300 (time and
    # probe error of each variant per problem); C selector and oracle rule
    # must pick the same variant for every swept problem and for off-grid
    # queries, under the pages' policy and under looser ones
    from fp8_precision_recommendation_gb300 import sweep
    rows = sweep.load_table(sweep.DEFAULT_TABLE)
    probs = sweep.problems()
    assert len(rows) == len(sweep.VARIANTS) * len(probs)
    for (m, n, k, norm, o) in probs:
        got = sorted(r[5] for r in rows if r[:5] == (m, n, k, norm, o))
        assert got == sorted(sweep.VARIANTS)
    for r in rows:
        assert r[6] > 0
        if r[5] == 3:
            assert r[7] == 0.0 and r[8] == 0.0
        else:
            assert 1e-3 < r[7] < 0.1          # E4M3 carries 3 mantissa bits
    table = [D.Entry(*r) for r in rows]
    queries = [p for p in probs] + [(65536, 256, 512, 1, 0.004), (8192, 1024, 2048, 1, 0.02),
                                    (524288, 64, 128, 1, 0.0), (100000, 256, 2048, 1, 0.01)]
    for pol in (D.Policy(1e-2, 0.2, -1.0), D.Policy(5e-2, -1.0, -1.0), D.Policy(5e-2, -1.0, 1.05)):
        for (m, n, k, norm, o) in queries:
            assert _c_select(table, m, n, k, norm, o, pol) == D.select(table, m, n, k, norm, o, pol)
