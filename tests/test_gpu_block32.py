"""GPU parity of square 32x32-block quantization (the GEM Training page's
[32, 32] block quantization): codes and E8M0 scales bit for bit against the
oracle, the transposed codes against the codes of the transpose, and the FP8
linear in this mode against the oracle by the rule in tests/parity.py."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import linear as OL
from oracle import probe as OP
from oracle import quantize as OQ
from parity import check_bf16_output

import fp8_precision_recommendation_gb300 as loka
from fp8_precision_recommendation_gb300 import _loka

pytestmark = pytest.mark.gpu

DEV = "cuda"
B32 = _loka.LOKA_SCALE_BLOCK32


def _gpu(t):
    return t.to(DEV) if t is not None else None


def _check(x_cpu, transposed=False, what=""):
    q, s, q_t = loka.quantize_fp8_block32(x_cpu.to(DEV), transposed=transposed)
    torch.cuda.synchronize()
    oq, os_ = OQ.quantize_block32(x_cpu)
    q, s = q.cpu().numpy(), s.cpu().numpy()
    assert np.array_equal(s, os_), f"{what}: {int((s != os_).sum())} scales differ"
    if not np.array_equal(q, oq):
        bad = np.argwhere(q != oq)[:6]
        raise AssertionError(f"{what}: {int((q != oq).sum())} codes differ; first "
                             f"{[(tuple(b), q[tuple(b)], oq[tuple(b)]) for b in bad]}")
    if transposed:
        assert np.array_equal(q_t.cpu().numpy(), q.T), f"{what}: transposed codes"
    return q, s


@pytest.mark.parametrize("rows,cols", [(32, 32), (64, 64), (70, 96), (1000, 512), (4096, 2080), (33, 4096)])
@pytest.mark.parametrize("dist", ["normal", "laplace"])
def test_block32_quantize_shapes(lib, rows, cols, dist):
    # ragged last block rows, a ragged last 256-column segment, long rows
    x = W.random_bf16((rows, cols), seed=rows + cols, dist=dist, outlier_frac=0.01)
    _check(x, what=f"{rows}x{cols} {dist}")


def test_block32_every_finite_bf16_pattern(lib):
    v = W.all_bf16_patterns()
    v = v[torch.isfinite(v.float())]
    v = v[: (v.numel() // 2048) * 2048].reshape(-1, 64)
    _check(v, what="all bf16")


def test_block32_zero_extreme_and_special_blocks(lib):
    x = torch.zeros((96, 96), dtype=torch.bfloat16)
    x[0, 0] = 3.0e38                       # a huge block
    x[40, 50] = 1e-40                      # a subnormal-only block
    x[70:, 70:] = -0.0
    x[33, 64:96] = torch.linspace(-5, 5, 32).to(torch.bfloat16)
    _check(x, transposed=True, what="special")


@pytest.mark.parametrize("rows,cols", [(64, 64), (256, 512), (1024, 96), (65536, 512)])
def test_block32_transposed_codes_are_the_codes_of_the_transpose(lib, rows, cols):
    x = W.random_bf16((rows, cols), seed=7 + rows, dist="laplace", outlier_frac=0.02)
    xd = x.to(DEV)
    q, s, q_t = loka.quantize_fp8_block32(xd, transposed=True)
    qT, sT, _ = loka.quantize_fp8_block32(xd.t().contiguous())
    torch.cuda.synchronize()
    assert torch.equal(q_t, q.t().contiguous())
    assert torch.equal(qT, q_t)
    assert torch.equal(sT, s.t().contiguous())


def test_block32_full_size_sampled_against_oracle(lib):
    inp = W.rec_mlp()
    q, s, q_t = loka.quantize_fp8_block32(inp.x.to(DEV), transposed=True)
    torch.cuda.synchronize()
    q, s = q.cpu().numpy(), s.cpu().numpy()
    rng = np.random.default_rng(3)
    for rb in np.unique(np.concatenate([[0, 1, inp.M // 32 - 1], rng.integers(0, inp.M // 32, 30)])):
        rows = slice(rb * 32, rb * 32 + 32)
        oq, os_ = OQ.quantize_block32(inp.x[rows])
        assert np.array_equal(q[rows], oq) and np.array_equal(s[rb:rb + 1], os_)
    assert torch.equal(q_t.cpu(), torch.from_numpy(q).t().contiguous())


def _layer(inp, **kw):
    return loka.Layer(x=_gpu(inp.x), w=_gpu(inp.w), bias=_gpu(inp.bias), gamma=_gpu(inp.gamma),
                      beta=_gpu(inp.beta), mode=inp.mode, norm=inp.norm, eps=inp.eps, **kw)


@pytest.mark.parametrize("N", [64, 192, 256, 512, 1024])
@pytest.mark.parametrize("norm", [W.NORM_NONE, W.NORM_LAYER, W.NORM_RMS])
def test_block32_linear_against_oracle(lib, N, norm):
    inp = W.make_layer(389, 256, N, mode=B32, norm=norm, seed=N + norm, x_dist="laplace", bias_var=0.02,
                       gamma_uniform=True)
    (y,) = loka.fp8_linear_norm([_layer(inp)])
    torch.cuda.synchronize()
    assert _loka.loka_device_status() == 0
    ye, _, _ = OL.linear_norm_inputs(inp)
    check_bf16_output(y.cpu(), ye, normalized=norm != W.NORM_NONE, what=f"block32 N{N} norm{norm}")


@pytest.mark.parametrize("K", [128, 512, 2048])
def test_block32_caller_quantized_inputs_match(lib, K):
    # the call quantizing bf16 X and W itself, and the caller handing it the
    # codes and scales of loka_quantize_fp8 (mode LOKA_SCALE_BLOCK32), give
    # the same bits
    inp = W.make_layer(700, K, 256, mode=B32, norm=W.NORM_LAYER, seed=K, bias_var=0.02, outlier_frac=0.01)
    (y_ref,) = loka.fp8_linear_norm([_layer(inp)])
    qx, sx = loka.quantize_fp8(_gpu(inp.x), B32)
    qw, sw = loka.quantize_fp8(_gpu(inp.w), B32)
    layer = loka.Layer(x=qx, x_scales=sx, w=qw, w_scales=sw, bias=_gpu(inp.bias), mode=B32, norm=W.NORM_LAYER,
                       eps=inp.eps)
    (y,) = loka.fp8_linear_norm([layer])
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_block32_probe_against_oracle(lib):
    inp = W.make_layer(512, 256, 256, mode=B32, norm=W.NORM_NONE, seed=5, bias_var=0.02, outlier_frac=0.01)
    got = loka.quant_error(_gpu(inp.x), _gpu(inp.w), _gpu(inp.bias), B32)
    ref = OP.quant_error(inp.x, inp.w, inp.bias, B32)
    assert got["count"] == ref["count"] and got["zero_ref_count"] == ref["zero_ref_count"]
    assert abs(got["rel_err_fro"] - ref["rel_err_fro"]) <= 1e-3 * ref["rel_err_fro"]
    assert abs(got["mere"] - ref["mere"]) <= 1e-2 * ref["mere"]
