"""GPU parity of the quantized output: the epilogue's E4M3 codes and scales of
its own bf16 output, handed to the next layer (quantization fused into the
preceding normalization, as on the GEM Training page).

Each case checks, on the same seeded inputs:
  * bit for bit: the codes and scales equal what loka_quantize_fp8 makes of
    the bf16 output of the same call (the unfused program);
  * against the oracle (linear_norm_quantized): the bf16 output meets the
    rule in tests/parity.py; the codes equal the oracle's wherever the two
    bf16 outputs and the row (or block) scales agree; every dequantized code
    lies within half an E4M3 step (at its scale) plus that bf16 tolerance of
    the exact normalized value (clipped to the largest code at that scale).
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import linear as OL
from parity import ULPS, check_bf16_output, to64

import fp8_precision_recommendation_gb300 as loka

pytestmark = pytest.mark.gpu

DEV = "cuda"
ROW, MX = W.SCALE_ROW, W.SCALE_MX32


def _gpu(t):
    return t.to(DEV) if t is not None else None


def _qlayer(inp, out_mode, y_q_only=False):
    return loka.Layer(x=_gpu(inp.x), w=_gpu(inp.w), bias=_gpu(inp.bias), gamma=_gpu(inp.gamma),
                      beta=_gpu(inp.beta), mode=inp.mode, norm=inp.norm, eps=inp.eps, y_q_mode=out_mode,
                      y_q_only=y_q_only)


def _run(layers):
    loka.fp8_linear_norm(layers)
    torch.cuda.synchronize()
    assert loka._loka.loka_device_status() == 0
    return layers


def _check_own_quantizer(layer, out_mode, what=""):
    """Codes and scales == loka_quantize_fp8 of the call's bf16 output."""
    q, s = loka.quantize_fp8(layer.y, out_mode)
    torch.cuda.synchronize()
    if not torch.equal(layer.y_q, q):
        bad = (layer.y_q != q).nonzero()[:6].tolist()
        raise AssertionError(f"{what}: {int((layer.y_q != q).sum())} codes differ from the quantizer; first "
                             f"{[(b, int(layer.y_q[b[0], b[1]]), int(q[b[0], b[1]])) for b in bad]}")
    if out_mode == ROW:
        assert torch.equal(layer.y_q_scales.view(torch.int32), s.view(torch.int32)), what
    else:
        assert torch.equal(layer.y_q_scales, s), what


def _element_scales(s, out_mode, N):
    """Per-element dequantization scale (float64) from row or block scales."""
    if out_mode == ROW:
        return np.repeat(s.astype(np.float64)[:, None], N, axis=1)
    return np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)


def _e4m3_half_step(a):
    """Half the E4M3 spacing at magnitude a (subnormal spacing below 2^-6)."""
    _, p = np.frexp(np.maximum(a, 2.0 ** -6))
    return np.ldexp(1.0, p - 1 - 3) / 2


def _check_oracle(inp, out_mode, layer, rows=None, what=""):
    y, yb, qo, so = OL.linear_norm_quantized_inputs(inp, out_mode, rows=rows)
    idx = slice(None) if rows is None else torch.as_tensor(rows)
    yg = layer.y[idx].cpu() if rows is not None else layer.y.cpu()
    normalized = inp.norm != W.NORM_NONE
    check_bf16_output(yg, y, normalized=normalized, what=what)
    qg = layer.y_q.cpu().numpy()
    sg = layer.y_q_scales.cpu().numpy()
    if rows is not None:
        qg, sg = qg[rows], sg[rows]
    N = qg.shape[1]
    ygf = to64(yg)
    if out_mode == ROW:
        same_scale = (sg.view(np.uint32) == np.asarray(so, np.float32).view(np.uint32))[:, None]
    else:
        same_scale = np.repeat(sg == so, 32, axis=1)
    same = same_scale & (ygf == yb)
    assert same.mean() > 0.5, f"{what}: only {same.mean():.2f} of the outputs agree with the oracle bit for bit"
    if not np.array_equal(qg[same], qo[same]):
        raise AssertionError(f"{what}: {int((qg[same] != qo[same]).sum())} codes differ where the bf16 outputs and "
                             f"scales agree")
    # dequantized codes against the exact value: half an E4M3 step at the
    # code's scale plus the bf16 output tolerance.  Codes saturate at +-448:
    # an MX block's largest elements may scale to just under 512, so the
    # reference is the exact value clipped to +-448 times the scale (the
    # clip moves two values no further apart)
    sc = _element_scales(sg, out_mode, N)
    dq = F.e4m3_decode(qg) * sc
    ref = np.clip(y, -448.0 * sc, 448.0 * sc)
    floor = 2.0 ** -6 if normalized else 2.0 ** -6 * np.sqrt(np.mean(y * y, axis=1, keepdims=True))
    tol = _e4m3_half_step(np.abs(ygf) / sc) * sc * (1 + 1e-9) + ULPS * F.bf16_ulp(np.maximum(np.abs(y), floor))
    err = np.abs(dq - ref)
    if (err > tol).any():
        i = np.argwhere(err > tol)[:5]
        raise AssertionError(f"{what}: {int((err > tol).sum())} dequantized codes beyond tolerance; first "
                             f"{[(tuple(k), dq[tuple(k)], y[tuple(k)]) for k in i]}")


def _case(M, K, N, mode, norm, affine, seed, x_dist="normal"):
    inp = W.make_layer(M, K, N, mode=mode, norm=norm, seed=seed, outlier_frac=0.01 if x_dist == "normal" else 0.0,
                       bias_var=0.02, gamma_uniform=affine, x_dist=x_dist,
                       eps=1e-6 if norm == W.NORM_RMS else 1e-5)
    if affine:
        inp.beta = W.random_bf16((N,), seed=seed + 1, var=0.1)
    return inp


@pytest.mark.parametrize("out_mode", [ROW, MX])
@pytest.mark.parametrize("norm", [W.NORM_NONE, W.NORM_LAYER, W.NORM_RMS])
@pytest.mark.parametrize("N", [64, 192, 256])
@pytest.mark.parametrize("affine", [False, True])
def test_small_shapes(lib, out_mode, norm, N, affine):
    # M spans several 128-row tiles and ends in a ragged tail
    inp = _case(389, 256, N, ROW, norm, affine, seed=N + 3 * norm + 11 * out_mode + 29 * affine)
    (layer,) = _run([_qlayer(inp, out_mode)])
    what = f"out{out_mode} norm{norm} N{N} affine{affine}"
    _check_own_quantizer(layer, out_mode, what)
    _check_oracle(inp, out_mode, layer, what=what)


@pytest.mark.parametrize("mode", [W.SCALE_TENSOR, W.SCALE_MX32])
@pytest.mark.parametrize("out_mode", [ROW, MX])
def test_other_input_scalings(lib, mode, out_mode):
    inp = _case(300, 512, 256, mode, W.NORM_LAYER, False, seed=40 + mode + 5 * out_mode)
    (layer,) = _run([_qlayer(inp, out_mode)])
    what = f"mode{mode} out{out_mode}"
    _check_own_quantizer(layer, out_mode, what)
    _check_oracle(inp, out_mode, layer, what=what)


@pytest.mark.parametrize("N", [512, 1024, 2048])
@pytest.mark.parametrize("mode,norm", [(ROW, W.NORM_LAYER), (W.SCALE_MX32, W.NORM_RMS)])
def test_cluster_wide_rows_mx_output(lib, N, mode, norm):
    # rows split over a cluster: every 32-column block is one CTA's
    inp = _case(300, 256, N, mode, norm, True, seed=N + mode, x_dist="laplace")
    (layer,) = _run([_qlayer(inp, MX)])
    what = f"cluster N{N} mode{mode}"
    _check_own_quantizer(layer, MX, what)
    _check_oracle(inp, MX, layer, what=what)


@pytest.mark.parametrize("out_mode", [ROW, MX])
@pytest.mark.parametrize("affine", [False, True])
def test_codes_without_the_bf16_copy(lib, out_mode, affine):
    inp = _case(700, 256, 256, ROW, W.NORM_LAYER, affine, seed=60 + out_mode + 2 * affine)
    (full,) = _run([_qlayer(inp, out_mode)])
    (only,) = _run([_qlayer(inp, out_mode, y_q_only=True)])
    assert only.y is None
    assert torch.equal(only.y_q, full.y_q)
    assert torch.equal(only.y_q_scales, full.y_q_scales)


def test_grouped_ragged_and_empty_groups(lib):
    inps = [_case(m, 256, 256, ROW, W.NORM_RMS, True, seed=70 + m) for m in (300, 0, 129, 1)]
    layers = _run([_qlayer(i, ROW) for i in inps])
    for inp, layer in zip(inps, layers):
        if inp.M:
            _check_own_quantizer(layer, ROW, f"group M{inp.M}")
            _check_oracle(inp, ROW, layer, what=f"group M{inp.M}")


@pytest.mark.parametrize("out_mode", [ROW, MX])
def test_two_layer_stack(lib, out_mode):
    # layer 2 takes layer 1's codes and scales as pre-quantized activations;
    # the same bits as layer 2 quantizing layer 1's bf16 output itself
    l1 = _case(1000, 512, 256, ROW, W.NORM_LAYER, False, seed=80 + out_mode)
    (a,) = _run([_qlayer(l1, out_mode)])
    w2 = _gpu(W.random_bf16((256, 256), seed=81, var=1.0 / 256))
    b2 = _gpu(W.random_bf16((256,), seed=82, var=0.02))
    stacked = loka.Layer(x=a.y_q, x_scales=a.y_q_scales, w=w2, bias=b2, mode=out_mode, norm=W.NORM_RMS, eps=1e-6)
    plain = loka.Layer(x=a.y, w=w2, bias=b2, mode=out_mode, norm=W.NORM_RMS, eps=1e-6)
    (y_stacked,) = loka.fp8_linear_norm([stacked])
    (y_plain,) = loka.fp8_linear_norm([plain])
    torch.cuda.synchronize()
    assert torch.equal(y_stacked.view(torch.int16), y_plain.view(torch.int16))


def test_special_rows(lib):
    # zero rows, subnormal inputs, huge values and Inf/NaN entries: the
    # codes and scales still equal the quantizer's on the bf16 output
    inp = _case(777, 512, 256, ROW, W.NORM_LAYER, False, seed=90)
    x = inp.x.clone()
    x[0] = 0
    x[5] = torch.tensor(2.0 ** -130, dtype=torch.float32).to(torch.bfloat16)
    x[6, ::7] = 1.0e15
    x[200, 3] = float("inf")
    x[201, 9] = float("nan")
    inp.x = x
    for out_mode in (ROW, MX):
        for norm in (W.NORM_NONE, W.NORM_LAYER):
            inp.norm = norm
            (layer,) = _run([_qlayer(inp, out_mode)])
            _check_own_quantizer(layer, out_mode, f"special out{out_mode} norm{norm}")


def test_rec_mlp_full_size(lib):
    inp = W.rec_mlp()
    (layer,) = _run([_qlayer(inp, ROW)])
    _check_own_quantizer(layer, ROW, "rec_mlp")
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(256), rng.integers(0, inp.M, 2048), np.arange(inp.M - 256, inp.M)]))
    _check_oracle(inp, ROW, layer, rows=rows, what="rec_mlp")


def test_mxfp8_layer_full_size(lib):
    inp = W.mxfp8()
    (layer,) = _run([_qlayer(inp, MX)])
    _check_own_quantizer(layer, MX, "mxfp8")
    rng = np.random.default_rng(6)
    rows = np.unique(np.concatenate([np.arange(128), rng.integers(0, inp.M, 512), np.arange(inp.M - 128, inp.M)]))
    _check_oracle(inp, MX, layer, rows=rows, what="mxfp8")
