"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle
on the same seeded inputs.  Quantized bytes and scales must be bit-exact;
bf16 outputs must meet the rule in tests/parity.py."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import linear as OL
from oracle import probe as OP
from oracle import quantize as OQ
from parity import check_bf16_output

import fp8_precision_recommendation_gb300 as loka
from fp8_precision_recommendation_gb300 import _loka

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _gpu(t):
    return t.to(DEV) if t is not None else None


def _oracle_quant(x, mode):
    q, s = OQ.quantize(x, mode)
    return q, np.asarray(s)


def _check_quant(x_cpu, mode, rows=None):
    q, s = loka.quantize_fp8(x_cpu.to(DEV), mode)
    torch.cuda.synchronize()
    q = q.cpu().numpy()
    s = s.cpu().numpy()
    if rows is not None:
        xq = x_cpu[torch.as_tensor(rows)]
        q = q[rows]
        s = s[rows] if mode != W.SCALE_TENSOR else s
    else:
        xq = x_cpu
    oq, os_ = _oracle_quant(xq, mode)
    if mode == W.SCALE_TENSOR:
        assert s.shape == (1,)
        assert np.float32(s[0]).tobytes() == np.float32(os_).tobytes()
    elif mode == W.SCALE_ROW:
        assert np.array_equal(s.view(np.uint32), os_.astype(np.float32).view(np.uint32))
    else:
        assert np.array_equal(s, os_)
    if not np.array_equal(q, oq):
        bad = np.argwhere(q != oq)[:8]
        raise AssertionError(f"{int((q != oq).sum())} codes differ; first {[(tuple(b), q[tuple(b)], oq[tuple(b)]) for b in bad]}")


# ------------------------------------------------------------ quantization
@pytest.mark.parametrize("mode", [W.SCALE_TENSOR, W.SCALE_ROW, W.SCALE_MX32])
def test_quantize_every_finite_bf16_pattern(lib, mode):
    v = W.all_bf16_patterns()
    fin = torch.isfinite(v.float())
    v = v[fin]
    v = v[: (v.numel() // 64) * 64].reshape(-1, 64)
    _check_quant(v, mode)


@pytest.mark.parametrize("mode", [W.SCALE_TENSOR, W.SCALE_ROW, W.SCALE_MX32])
def test_quantize_every_bf16_pattern_at_unit_scale(lib, mode):
    # rows whose amax is 448 (tensor/row) so that x * inv == x exactly, or MX
    # blocks whose scale is 2^0, put every bf16 value through the cast itself
    v = W.all_bf16_patterns().float()
    fin = torch.isfinite(v) & (v.abs() <= 448)
    v = v[fin]
    n = (v.numel() // 31) * 31
    body = v[:n].reshape(-1, 31)
    anchor = torch.full((body.shape[0], 1), 448.0 if mode != W.SCALE_MX32 else 256.0)
    x = torch.cat([anchor, body], dim=1).to(torch.bfloat16)
    x = torch.cat([x, x], dim=1)      # 64 columns (two MX blocks)
    _check_quant(x, mode)


@pytest.mark.parametrize("mode", [W.SCALE_ROW, W.SCALE_MX32])
@pytest.mark.parametrize("cols", [32, 64, 96, 128, 160, 256, 512, 1024, 2048, 2080, 4096])
def test_quantize_shapes_and_ragged_widths(lib, mode, cols):
    x = W.random_bf16((37, cols), seed=cols, dist="laplace", outlier_frac=0.01)
    _check_quant(x, mode)


def test_quantize_row_scale_for_every_bf16_amax(lib):
    # one row per positive finite bf16 magnitude, that value as the row's
    # only non-zero entry: every mantissa at every exponent (subnormal and
    # tiny amax included) goes through the row-scale computation
    pats = torch.arange(1, 0x7F80, dtype=torch.int32).to(torch.int16)
    v = pats.view(torch.bfloat16)
    x = torch.zeros((v.numel(), 32), dtype=torch.bfloat16)
    x[:, 0] = v
    x[::2, 5] = -v[::2]          # the negative twin in half of the rows
    _check_quant(x, W.SCALE_ROW)


def test_quantize_zero_and_extreme_rows(lib):
    x = torch.zeros((6, 64), dtype=torch.bfloat16)
    x[1, 3] = 1e-38
    x[2, 5] = -3.0e38
    x[3, :] = -0.0
    x[4, 7] = 1e-40          # bf16 subnormal
    x[5, 0] = 3.0e38
    x[5, 1] = 1.0
    for mode in (W.SCALE_TENSOR, W.SCALE_ROW, W.SCALE_MX32):
        _check_quant(x, mode)


def test_quantize_infinite_inputs(lib):
    # amax = inf: rowwise gives inv = 0, so finite elements become signed
    # zeros and the infinity becomes a NaN code (sign unspecified); MX gives
    # the block exponent of 2^128 and the infinity saturates to 448.
    x = torch.ones((2, 64), dtype=torch.bfloat16)
    x[0, 3] = float("inf")
    x[1, 5] = -float("inf")
    x[1, 6] = -2.0
    q, s = loka.quantize_fp8(x.to(DEV), W.SCALE_ROW)
    q = q.cpu().numpy()
    assert np.isinf(s.cpu().numpy()).all()
    assert q[0, 3] & 0x7F == 0x7F and q[1, 5] & 0x7F == 0x7F
    assert q[0, 0] == 0x00 and q[1, 6] == 0x80
    q, s = loka.quantize_fp8(x.to(DEV), W.SCALE_MX32)
    q, s = q.cpu().numpy(), s.cpu().numpy()
    assert q[0, 3] == 0x7E and q[1, 5] == 0xFE
    oq, os_ = OQ.quantize_mx(x)
    assert np.array_equal(q, oq) and np.array_equal(s, os_)


@pytest.mark.parametrize("mode", [W.SCALE_TENSOR, W.SCALE_ROW, W.SCALE_MX32])
def test_quantize_single_config_bit_exact(lib, mode):
    inp = W.single()
    _check_quant(inp.x, mode)
    _check_quant(inp.w, mode)


def test_quantize_rec_mlp_full_size_rowwise(lib):
    inp = W.rec_mlp()
    _check_quant(inp.x, W.SCALE_ROW)
    _check_quant(inp.w, W.SCALE_ROW)


def test_quantize_mxfp8_layer_sampled_rows(lib):
    inp = W.mxfp8()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(128), rng.integers(0, inp.M, 2048), np.arange(inp.M - 128, inp.M)]))
    _check_quant(inp.x, W.SCALE_MX32, rows=rows)
    _check_quant(inp.w, W.SCALE_MX32)


@pytest.mark.parametrize("mode", [W.SCALE_TENSOR, W.SCALE_ROW, W.SCALE_MX32, W.SCALE_BLOCK32])
def test_quantize_strided_column_slice(lib, mode):
    # x is a column slice of a wider tensor: rows start ld = 520 elements
    # apart; the codes and scales are those of the dense copy of the slice
    wide = W.random_bf16((300, 520), seed=31, dist="laplace", outlier_frac=0.01)
    view = wide.to(DEV)[:, 136:392]
    assert view.stride(0) == 520 and not view.is_contiguous()
    rows, cols = view.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=DEV)
    shp, dt = loka.scales_shape(rows, cols, mode)
    s = torch.empty(shp, dtype=getattr(torch, dt), device=DEV)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    _loka.loka_quantize_fp8(view, rows, cols, 520, mode, q, s, ws, 256)
    torch.cuda.synchronize()
    oq, os_ = _oracle_quant(wide[:, 136:392].contiguous(), mode)
    assert np.array_equal(q.cpu().numpy(), oq)
    got = s.cpu().numpy()
    if mode in (W.SCALE_TENSOR, W.SCALE_ROW):
        assert np.array_equal(got.reshape(-1).view(np.uint32), np.asarray(os_, np.float32).reshape(-1).view(np.uint32))
    else:
        assert np.array_equal(got, os_)


def test_quantize_empty(lib):
    q = torch.empty((0, 64), dtype=torch.uint8, device=DEV)
    s = torch.zeros((1,), dtype=torch.float32, device=DEV)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    _loka.loka_quantize_fp8(x, 0, 64, 64, W.SCALE_TENSOR, q, s, ws, 256)
    torch.cuda.synchronize()
    assert s.item() == 1.0


# ------------------------------------------------------- linear + norm
def _layer(inp, y=None):
    return loka.Layer(x=_gpu(inp.x), w=_gpu(inp.w), bias=_gpu(inp.bias), gamma=_gpu(inp.gamma),
                      beta=_gpu(inp.beta), mode=inp.mode, norm=inp.norm, eps=inp.eps, y=y)


def _run(inps):
    ys = loka.fp8_linear_norm([_layer(i) for i in inps])
    torch.cuda.synchronize()
    assert loka._loka.loka_device_status() == 0
    return [y.cpu() for y in ys]


def _check_layer(inp, y_gpu, rows=None, what=""):
    y, _, _ = OL.linear_norm_inputs(inp, rows=rows)
    g = y_gpu if rows is None else y_gpu[torch.as_tensor(rows)]
    return check_bf16_output(g, y, normalized=inp.norm != W.NORM_NONE, what=what)


def test_single_config_per_tensor_layernorm(lib):
    inp = W.single()
    (y,) = _run([inp])
    _check_layer(inp, y, what="single")


@pytest.mark.parametrize("mode", [W.SCALE_TENSOR, W.SCALE_ROW, W.SCALE_BF16])
@pytest.mark.parametrize("norm", [W.NORM_NONE, W.NORM_LAYER, W.NORM_RMS])
@pytest.mark.parametrize("N", [64, 128, 192, 256, 512])
def test_small_shapes_all_variants(lib, mode, norm, N):
    # M spans several 128-row tiles and ends in a ragged tail
    inp = W.make_layer(389, 256, N, mode=mode, norm=norm, seed=N + 7 * norm + 31 * mode,
                       outlier_frac=0.01, bias_var=0.02, gamma_uniform=True)
    inp.beta = W.random_bf16((N,), seed=5, var=0.1)
    (y,) = _run([inp])
    _check_layer(inp, y, what=f"mode{mode} norm{norm} N{N}")


@pytest.mark.parametrize("M", [1, 127, 128, 129, 1000])
@pytest.mark.parametrize("K", [128, 384, 2048])
def test_ragged_m_and_k(lib, M, K):
    inp = W.make_layer(M, K, 256, mode=W.SCALE_ROW, norm=W.NORM_LAYER, seed=M + K, bias_var=0.02)
    (y,) = _run([inp])
    _check_layer(inp, y, what=f"M{M} K{K}")


def test_m_zero_is_a_no_op(lib):
    inp = W.make_layer(0, 128, 128, mode=W.SCALE_ROW, norm=W.NORM_LAYER)
    (y,) = _run([inp])
    assert y.shape == (0, 128)


def test_rec_mlp_full_size(lib):
    inp = W.rec_mlp()
    (y,) = _run([inp])
    _check_layer(inp, y, what="rec_mlp (every row)")
    # properties of every row: LayerNorm output has mean ~0 and mean square ~1
    yf = y.float()
    assert yf.mean(dim=1).abs().max().item() < 2e-2
    assert (yf.pow(2).mean(dim=1) - 1).abs().max().item() < 2e-2


def test_ensemble_grouped_launch(lib):
    inps = W.ensemble()
    ys = _run(inps)
    for g, (inp, y) in enumerate(zip(inps, ys)):
        _check_layer(inp, y, what=f"group{g} (every row)")


# LoKA section III-B ("Normalization overhead and errors") names mean
# cancellation as LayerNorm's weakness: rows whose mean lies far above their
# spread.  A bias of ratio x (the spread of Wx is about 1) puts every row's
# mean ratio times above its standard deviation; the exact oracle shows any
# loss of the small signal at once.
@pytest.mark.parametrize("ratio", [1e2, 1e3, 1e4])
@pytest.mark.parametrize("mode,N", [(W.SCALE_ROW, 256), (W.SCALE_MX32, 256), (W.SCALE_ROW, 2048),
                                    (W.SCALE_MX32, 2048)])
def test_layernorm_mean_cancellation_bias_offset(lib, ratio, mode, N):
    inp = W.make_layer(389, 256, N, mode=mode, norm=W.NORM_LAYER, seed=int(ratio) + N + mode, bias_var=0.02,
                       gamma_uniform=True, outlier_frac=0.01)
    inp.bias = (inp.bias.float() + ratio).to(torch.bfloat16)
    inp.beta = W.random_bf16((N,), seed=12, var=0.1)
    (y,) = _run([inp])
    _check_layer(inp, y, what=f"bias offset {ratio:g} mode{mode} N{N}")


# The same regime with the offset inside the accumulator: a constant column
# of X meets a constant column of W, so every output of a row carries the
# product before the bias is added.  The fp32 accumulator itself rounds
# that running sum once per 32-wide K step, each time by up to half an fp32
# ulp of the offset in code units, which no epilogue can undo.  At 10^2
# that stays far inside the 2-ulp rule; at 10^3 the rule gets that
# allowance on top: (K/32) * ulp_fp32(|offset|) * rstd (a whole ulp per step:
# the dequantization scale moves the offset by up to a factor of two against
# its binade in code units), the offset and rstd of each row taken from the
# exact oracle.
def _in_accumulator_layer(ratio, mode, N):
    inp = W.make_layer(389, 256, N, mode=mode, norm=W.NORM_LAYER, seed=int(ratio) + 3 * N, bias_var=0.02)
    x = inp.x.clone()
    w = inp.w.clone()
    x[:, 0] = ratio
    w[:, 0] = 1.0
    inp.x, inp.w = x, w
    return inp


@pytest.mark.parametrize("mode,N", [(W.SCALE_ROW, 256), (W.SCALE_MX32, 512)])
def test_layernorm_mean_cancellation_in_accumulator(lib, mode, N):
    inp = _in_accumulator_layer(1e2, mode, N)
    (y,) = _run([inp])
    _check_layer(inp, y, what=f"accumulator offset 1e2 mode{mode} N{N}")


@pytest.mark.parametrize("mode,N", [(W.SCALE_ROW, 256), (W.SCALE_MX32, 512)])
def test_layernorm_mean_cancellation_in_accumulator_fp32_bound(lib, mode, N):
    from oracle.formats import bf16_ulp
    inp = _in_accumulator_layer(1e3, mode, N)
    (y,) = _run([inp])
    y_exact, _, _ = OL.linear_norm_inputs(inp)
    v, _ = OL.prenorm(inp.x, inp.w, inp.bias, mode)
    b = OL.vec64(inp.bias, N, 0.0)
    off = np.abs(v - b[None, :]).max(axis=1, keepdims=True)          # the row's offset inside the accumulator
    rstd = 1.0 / np.sqrt(v.var(axis=1, keepdims=True) + inp.eps)
    ulp32 = np.exp2(np.floor(np.log2(off)) - 23)
    allowance = (inp.K / 32) * ulp32 * rstd
    g = y.to(torch.float64).numpy()
    tol = 2 * bf16_ulp(np.maximum(np.abs(y_exact), 2.0 ** -6)) + allowance
    err = np.abs(g - y_exact)
    assert (err <= tol).all(), f"{int((err > tol).sum())} elements beyond 2 ulps + the fp32 accumulation allowance"


def test_grouped_with_ragged_and_empty_groups(lib):
    inps = [W.make_layer(m, 256, 256, mode=W.SCALE_ROW, norm=W.NORM_RMS, seed=m, gamma_uniform=True, eps=1e-6)
            for m in (300, 0, 129, 1)]
    ys = _run(inps)
    for inp, y in zip(inps, ys):
        if inp.M:
            _check_layer(inp, y, what=f"M{inp.M}")


def test_prequantized_inputs_match_bf16_inputs(lib):
    inp = W.make_layer(500, 512, 256, mode=W.SCALE_ROW, norm=W.NORM_LAYER, seed=3, bias_var=0.02, outlier_frac=0.01)
    (y_ref,) = _run([inp])
    x, w = _gpu(inp.x), _gpu(inp.w)
    qx, sx = loka.quantize_fp8(x, W.SCALE_ROW)
    qw, sw = loka.quantize_fp8(w, W.SCALE_ROW)
    layer = loka.Layer(x=qx, w=qw, x_scales=sx, w_scales=sw, bias=_gpu(inp.bias), mode=W.SCALE_ROW,
                       norm=W.NORM_LAYER, eps=inp.eps)
    (y,) = loka.fp8_linear_norm([layer])
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), y_ref)


def _two_step(inps):
    """The same layers with X and W quantized by loka_quantize_fp8 first and
    handed to the GEMM as E4M3."""
    layers = []
    for inp in inps:
        x, w = _gpu(inp.x), _gpu(inp.w)
        qx, sx = loka.quantize_fp8(x, inp.mode)
        qw, sw = loka.quantize_fp8(w, inp.mode)
        layers.append(loka.Layer(x=qx, w=qw, x_scales=sx, w_scales=sw, bias=_gpu(inp.bias), gamma=_gpu(inp.gamma),
                                 beta=_gpu(inp.beta), mode=inp.mode, norm=inp.norm, eps=inp.eps))
    ys = loka.fp8_linear_norm(layers)
    torch.cuda.synchronize()
    return [y.cpu() for y in ys]


@pytest.mark.parametrize("K", [32, 64, 128, 256, 512])
@pytest.mark.parametrize("N", [64, 128, 192, 256])
@pytest.mark.parametrize("norm", [W.NORM_NONE, W.NORM_LAYER, W.NORM_RMS])
def test_bf16_inputs_match_caller_quantized_inputs(lib, K, N, norm):
    # the call with bf16 X and W quantizes them itself; handing it the
    # codes and scales of loka_quantize_fp8 must give the same bits
    inps = [W.make_layer(m, K, N, mode=W.SCALE_ROW, norm=norm, seed=m + K + N, bias_var=0.02, outlier_frac=0.01,
                         gamma_uniform=True, eps=1e-5 if norm != W.NORM_RMS else 1e-6)
            for m in (1000, 129, 1)]
    ys = _run(inps)
    ref = _two_step(inps)
    for inp, y, r in zip(inps, ys, ref):
        assert torch.equal(y.view(torch.int16), r.view(torch.int16)), f"M={inp.M}"
    _check_layer(inps[0], ys[0], what="oracle")


def test_special_rows_through_the_layer(lib):
    # zero rows (scale 1), rows of subnormals, huge values, and Inf/NaN
    # entries: the same bits with caller- and library-quantized inputs, the
    # oracle on the finite rows, NaN rows where X holds Inf or NaN
    inp = W.make_layer(777, 512, 256, mode=W.SCALE_ROW, norm=W.NORM_LAYER, seed=11, bias_var=0.02)
    x = inp.x.clone()
    x[0] = 0
    x[5] = torch.tensor(2.0 ** -130, dtype=torch.float32).to(torch.bfloat16)
    x[6, ::7] = 1.0e15
    x[200, 3] = float("inf")
    x[201, 9] = float("nan")
    x[776] = -x[776]
    inp.x = x
    (y,) = _run([inp])
    (r,) = _two_step([inp])
    assert torch.equal(y.view(torch.int16), r.view(torch.int16))
    assert torch.isnan(y[200:202].float()).all()
    ok = [m for m in range(inp.M) if m not in (200, 201)]
    _check_layer(inp, y, rows=np.array(ok[:64] + ok[-64:]), what="finite rows")


def test_deterministic(lib):
    inp = W.make_layer(1000, 512, 256, mode=W.SCALE_ROW, norm=W.NORM_LAYER, seed=4, bias_var=0.02)
    (a,) = _run([inp])
    (b,) = _run([inp])
    assert torch.equal(a, b)


# ----------------------------------------------------------------- probe
@pytest.mark.parametrize("mode", [W.SCALE_TENSOR, W.SCALE_ROW, W.SCALE_BF16])
def test_quant_error_probe_matches_oracle(lib, mode):
    inp = W.make_layer(1000, 512, 256, mode=mode, norm=W.NORM_NONE, seed=6, bias_var=0.02, outlier_frac=0.01)
    st = loka.quant_error(_gpu(inp.x), _gpu(inp.w), _gpu(inp.bias), mode)
    want = OP.quant_error(inp.x, inp.w, inp.bias, mode)
    assert st["count"] == want["count"]
    assert st["zero_ref_count"] == want["zero_ref_count"]
    if mode == W.SCALE_BF16:
        assert st["rel_err_fro"] < 1e-6 and st["mere"] < 1e-5
    else:
        assert abs(st["rel_err_fro"] - want["rel_err_fro"]) <= 1e-3 * want["rel_err_fro"]
        assert abs(st["mere"] - want["mere"]) <= 1e-2 * want["mere"]
        assert abs(st["max_abs"] - want["max_abs"]) <= 1e-3 * want["max_abs"] + 1e-6


@pytest.mark.parametrize("mode,norm,act", [(W.SCALE_ROW, W.NORM_LAYER, 0), (W.SCALE_MX32, W.NORM_RMS, 0),
                                           (W.SCALE_TENSOR, W.NORM_LAYER, 1)])
def test_quant_error_post_norm_matches_oracle(lib, mode, norm, act):
    inp = W.make_layer(700, 512, 256, mode=mode, norm=norm, seed=9 + mode, bias_var=0.02, outlier_frac=0.01,
                       gamma_uniform=True)
    beta = W.random_bf16((256,), seed=4, var=0.1) if norm == W.NORM_LAYER else None
    st = loka.quant_error(_gpu(inp.x), _gpu(inp.w), _gpu(inp.bias), mode, norm=norm, eps=inp.eps,
                          gamma=_gpu(inp.gamma), beta=_gpu(beta), act=act)
    want = OP.quant_error(inp.x, inp.w, inp.bias, mode, norm=norm, gamma=inp.gamma, beta=beta, eps=inp.eps, act=act)
    # both sides' post-norm outputs carry fp32 rounding (statistics, rsqrt)
    assert abs(st["max_abs_post_norm"] - want["max_abs_post_norm"]) <= 1e-3 * want["max_abs_post_norm"] + 1e-5
    assert abs(st["rel_err_fro"] - want["rel_err_fro"]) <= 1e-3 * want["rel_err_fro"]


# -------------------------------------------------------------- watchdog
def test_watchdog_turns_a_stuck_wait_into_a_status(lib):
    assert _loka.loka_device_status() == _loka.LOKA_OK
    _loka.loka_selftest_watchdog(2_000_000)          # 2 ms
    assert _loka.loka_device_status() == _loka.LOKA_ERR_TIMEOUT
    assert _loka.loka_device_status() == _loka.LOKA_OK   # cleared, context still usable
    inp = W.single()
    (y,) = _run([inp])
    _check_layer(inp, y, what="after watchdog")


def test_tensor_peak_microbenchmark(lib):
    # the tcgen05 peak the contraction's tensor-pipe share is measured
    # against: both kinds complete with a clean status, and E4M3 (K = 32 per
    # MMA) runs at least 1.5x the bf16 FLOP rate (K = 16 in the same time)
    dev = torch.device(DEV)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rate = {}
    for kind, k in ((0, 32), (1, 16)):
        _loka.loka_selftest_mma_peak(kind, 1024)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        _loka.loka_selftest_mma_peak(kind, 100_000)
        b.record()
        b.synchronize()
        rate[kind] = sms * 100_000 * 2.0 * 128 * 256 * k / (a.elapsed_time(b) / 1e3)
    assert _loka.loka_device_status() == _loka.LOKA_OK
    assert rate[0] > 1.5 * rate[1] > 0
    with pytest.raises(_loka.LokaError):
        _loka.loka_selftest_mma_peak(2, 1)
    with pytest.raises(_loka.LokaError):
        _loka.loka_selftest_mma_peak(0, 0)


# -------------------------------------------------------------- MX 1x32
@pytest.mark.parametrize("N", [64, 128, 192, 256])
@pytest.mark.parametrize("norm", [W.NORM_NONE, W.NORM_LAYER, W.NORM_RMS])
def test_mx_block_scaled_small_shapes(lib, N, norm):
    inp = W.make_layer(389, 256, N, mode=W.SCALE_MX32, norm=norm, seed=N + 3 * norm, x_dist="laplace",
                       outlier_frac=0.01, bias_var=0.02, gamma_uniform=True)
    (y,) = _run([inp])
    _check_layer(inp, y, what=f"MX norm{norm} N{N}")


def test_mx_scales_vary_per_row_and_block(lib):
    # rows and 32-element blocks with very different magnitudes, so that a
    # scale code applied to the wrong row or block shows up at once
    M, K, N = 256, 512, 128
    rng = np.random.default_rng(7)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-12, 12, size=(M, K // 32))).repeat(32, axis=1).astype(np.float32)
    w = (rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)
    w *= np.exp2(rng.integers(-6, 6, size=(N, K // 32))).repeat(32, axis=1).astype(np.float32)
    inp = W.LayerInputs(x=torch.from_numpy(x).to(torch.bfloat16), w=torch.from_numpy(w).to(torch.bfloat16),
                        bias=None, gamma=None, beta=None, mode=W.SCALE_MX32, norm=W.NORM_NONE, eps=0.0)
    (y,) = _run([inp])
    _check_layer(inp, y, what="MX structured scales")


def test_mx_long_k_layer(lib):
    inp = W.make_layer(4096, 2048, 256, mode=W.SCALE_MX32, norm=W.NORM_LAYER, seed=5, x_dist="laplace")
    (y,) = _run([inp])
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([np.arange(128), rng.integers(0, inp.M, 512), np.arange(inp.M - 128, inp.M)]))
    _check_layer(inp, y, rows=rows, what="MX K=2048")


def test_mx_prequantized_inputs_match_bf16_inputs(lib):
    inp = W.make_layer(300, 256, 128, mode=W.SCALE_MX32, norm=W.NORM_RMS, seed=8, x_dist="laplace", eps=1e-6)
    (y_ref,) = _run([inp])
    qx, sx = loka.quantize_fp8(_gpu(inp.x), W.SCALE_MX32)
    qw, sw = loka.quantize_fp8(_gpu(inp.w), W.SCALE_MX32)
    layer = loka.Layer(x=qx, w=qw, x_scales=sx, w_scales=sw, mode=W.SCALE_MX32, norm=W.NORM_RMS, eps=inp.eps)
    (y,) = loka.fp8_linear_norm([layer])
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), y_ref)


def test_mx_probe_matches_oracle(lib):
    inp = W.make_layer(1000, 512, 256, mode=W.SCALE_MX32, norm=W.NORM_NONE, seed=6, bias_var=0.02, x_dist="laplace")
    st = loka.quant_error(_gpu(inp.x), _gpu(inp.w), _gpu(inp.bias), W.SCALE_MX32)
    want = OP.quant_error(inp.x, inp.w, inp.bias, W.SCALE_MX32)
    assert abs(st["rel_err_fro"] - want["rel_err_fro"]) <= 1e-3 * want["rel_err_fro"]
    assert abs(st["mere"] - want["mere"]) <= 1e-2 * want["mere"]


# ------------------------------------------- rows wider than one CTA (clusters)
@pytest.mark.parametrize("N", [512, 1024, 2048])
@pytest.mark.parametrize("mode,norm", [(W.SCALE_ROW, W.NORM_LAYER), (W.SCALE_MX32, W.NORM_RMS),
                                       (W.SCALE_TENSOR, W.NORM_NONE), (W.SCALE_MX32, W.NORM_LAYER)])
def test_cluster_wide_rows(lib, N, mode, norm):
    inp = W.make_layer(300, 256, N, mode=mode, norm=norm, seed=N + mode, x_dist="laplace",
                       bias_var=0.02, gamma_uniform=True)
    inp.beta = W.random_bf16((N,), seed=9, var=0.1)
    (y,) = _run([inp])
    _check_layer(inp, y, what=f"cluster N{N} mode{mode} norm{norm}")


def test_cluster_grouped_ragged(lib):
    inps = [W.make_layer(m, 256, 512, mode=W.SCALE_ROW, norm=W.NORM_LAYER, seed=m, bias_var=0.02) for m in (129, 0, 400)]
    ys = _run(inps)
    for inp, y in zip(inps, ys):
        if inp.M:
            _check_layer(inp, y, what=f"cluster group M{inp.M}")


def test_mxfp8_layer_full_size(lib):
    inp = W.mxfp8()
    (y,) = _run([inp])
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([np.arange(128), rng.integers(0, inp.M, 1024), np.arange(inp.M - 128, inp.M)]))
    _check_layer(inp, y, rows=rows, what="mxfp8 262144x2048x512")
    yf = y.float()
    assert yf.mean(dim=1).abs().max().item() < 2e-2
    assert (yf.pow(2).mean(dim=1) - 1).abs().max().item() < 2e-2


def test_variant_sweep_smoke(lib):
    # the sweep that writes the dispatch table: every variant timed and its
    # probe error measured on two small problems
    from fp8_precision_recommendation_gb300 import sweep
    table = sweep.run(quick=True, log=lambda *a: None)
    rows = table["rows"]
    assert len(rows) == len(sweep.VARIANTS) * len(sweep.problems(quick=True))
    for (m, n, k, norm, o, v, t, rel, mere) in rows:
        assert t > 0
        if v == _loka.LOKA_BF16:
            assert rel == 0.0
        else:
            assert 1e-3 < rel < 0.1


# ------------------------------------------------- general layer shapes
# Any K and N that are multiples of 32 (LoKA section II-C's production GEMM
# shapes are not all multiples of 128): the last K slice reads zeros past K;
# rows narrower than the kernel's columns skip the empty chunks; rows wider
# than a CTA split over 256-column CTAs, the last one partial or empty.
@pytest.mark.parametrize("K", [32, 64, 96, 160, 320])
@pytest.mark.parametrize("mode", [W.SCALE_TENSOR, W.SCALE_ROW, W.SCALE_MX32, W.SCALE_BF16, W.SCALE_BLOCK32])
def test_k_multiple_of_32(lib, K, mode):
    inp = W.make_layer(389, K, 256, mode=mode, norm=W.NORM_LAYER, seed=K + 11 * mode, outlier_frac=0.01,
                       bias_var=0.02, gamma_uniform=True)
    (y,) = _run([inp])
    _check_layer(inp, y, what=f"K{K} mode{mode}")


@pytest.mark.parametrize("N", [32, 96, 160, 224])
@pytest.mark.parametrize("mode,norm", [(W.SCALE_ROW, W.NORM_LAYER), (W.SCALE_MX32, W.NORM_RMS),
                                       (W.SCALE_TENSOR, W.NORM_NONE), (W.SCALE_BF16, W.NORM_LAYER)])
def test_narrow_n_multiple_of_32(lib, N, mode, norm):
    inp = W.make_layer(300, 256, N, mode=mode, norm=norm, seed=N + 5 * mode, outlier_frac=0.01,
                       bias_var=0.02, gamma_uniform=True)
    inp.beta = W.random_bf16((N,), seed=3, var=0.1)
    (y,) = _run([inp])
    _check_layer(inp, y, what=f"N{N} mode{mode} norm{norm}")


@pytest.mark.parametrize("N", [320, 768, 1056, 2016])
@pytest.mark.parametrize("mode,norm", [(W.SCALE_ROW, W.NORM_LAYER), (W.SCALE_MX32, W.NORM_RMS),
                                       (W.SCALE_ROW, W.NORM_NONE), (W.SCALE_MX32, W.NORM_LAYER)])
def test_wide_n_multiple_of_32(lib, N, mode, norm):
    inp = W.make_layer(200, 128, N, mode=mode, norm=norm, seed=N + 7 * mode + norm, x_dist="laplace",
                       bias_var=0.02, gamma_uniform=True)
    inp.beta = W.random_bf16((N,), seed=4, var=0.1)
    (y,) = _run([inp])
    _check_layer(inp, y, what=f"N{N} mode{mode} norm{norm}")


@pytest.mark.parametrize("N", [96, 320])
def test_odd_width_blocknorm_and_quantized_output(lib, N):
    # BlockNorm over 32-column blocks on a partial CTA, and E4M3 output rows
    # (per-row output scales need N <= 256; MX scales any width)
    inp = W.make_layer(257, 96, N, mode=W.SCALE_ROW, norm=W.NORM_BLOCK_RMS, seed=N, outlier_frac=0.01,
                       bias_var=0.02, gamma_uniform=True)
    inp.norm_block = 32

    def lay(out_mode=None):
        return loka.Layer(x=_gpu(inp.x), w=_gpu(inp.w), bias=_gpu(inp.bias), gamma=_gpu(inp.gamma),
                          beta=_gpu(inp.beta), mode=inp.mode, norm=inp.norm, eps=inp.eps, norm_block=32,
                          y_q_mode=out_mode)

    (y,) = loka.fp8_linear_norm([lay()])
    torch.cuda.synchronize()
    assert loka._loka.loka_device_status() == 0
    _check_layer(inp, y.cpu(), what=f"BlockNorm N{N}")
    for out_mode in ([W.SCALE_ROW, W.SCALE_MX32] if N <= 256 else [W.SCALE_MX32]):
        layer = lay(out_mode)
        loka.fp8_linear_norm([layer])
        torch.cuda.synchronize()
        assert torch.equal(layer.y.cpu(), y.cpu())
        q, s = loka.quantize_fp8(layer.y, out_mode)
        torch.cuda.synchronize()
        assert torch.equal(layer.y_q, q), f"N{N} out{out_mode}"
        assert torch.equal(layer.y_q_scales.view(torch.uint8), s.view(torch.uint8)), f"N{N} out{out_mode}"


# ------------------------------------------------ a partial last wave
# Row counts that leave the persistent grid's last wave a quarter full, the
# last tile ragged (both 64-row halves partly filled, the second half empty,
# or full): every row against the oracle, for the per-row, MX, bf16 and
# BlockNorm epilogues and the quantized outputs.
def _tail_rows(tail):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = sms + sms // 4
    return (tiles - 1) * 128 + tail


@pytest.mark.parametrize("tail", [111, 30, 128])
@pytest.mark.parametrize("mode,norm", [(W.SCALE_ROW, W.NORM_LAYER), (W.SCALE_MX32, W.NORM_RMS),
                                       (W.SCALE_ROW, W.NORM_BLOCK_RMS), (W.SCALE_BF16, W.NORM_LAYER)])
def test_partial_last_wave(lib, tail, mode, norm):
    M = _tail_rows(tail)
    inp = W.make_layer(M, 512, 256, mode=mode, norm=norm, seed=tail + 3 * mode + norm, outlier_frac=0.01,
                       bias_var=0.02, gamma_uniform=True)
    if norm == W.NORM_BLOCK_RMS:
        inp.norm_block = 64
        layer = loka.Layer(x=_gpu(inp.x), w=_gpu(inp.w), bias=_gpu(inp.bias), gamma=_gpu(inp.gamma),
                           mode=inp.mode, norm=inp.norm, eps=inp.eps, norm_block=64)
        (y,) = loka.fp8_linear_norm([layer])
        torch.cuda.synchronize()
        y = y.cpu()
    else:
        (y,) = _run([inp])
    _check_layer(inp, y, what=f"M{M} mode{mode} norm{norm} (every row)")


def test_partial_last_wave_quantized_output(lib):
    M = _tail_rows(77)
    inp = W.make_layer(M, 512, 256, mode=W.SCALE_ROW, norm=W.NORM_LAYER, seed=77, outlier_frac=0.01, bias_var=0.02)
    for out_mode in (W.SCALE_ROW, W.SCALE_MX32):
        layer = loka.Layer(x=_gpu(inp.x), w=_gpu(inp.w), bias=_gpu(inp.bias), mode=inp.mode, norm=inp.norm,
                           eps=inp.eps, y_q_mode=out_mode)
        loka.fp8_linear_norm([layer])
        torch.cuda.synchronize()
        assert loka._loka.loka_device_status() == 0
        _check_layer(inp, layer.y.cpu(), what=f"M{M} quantized out {out_mode}")
        q, s = loka.quantize_fp8(layer.y, out_mode)
        torch.cuda.synchronize()
        assert torch.equal(layer.y_q, q) and torch.equal(layer.y_q_scales.view(torch.uint8), s.view(torch.uint8))
