"""GPU parity of BlockNorm (LoKA section III-B 2: RMSNorm over fixed blocks
of the output row) and Hard Swish (section III-B 3) in the GEMM epilogue,
against the oracle on the same seeded inputs: bf16 outputs by the rule in
tests/parity.py, E4M3 outputs bit for bit against the library's quantizer on
the same call's bf16 output and against the oracle as in
test_gpu_quantized_output."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import linear as OL
from parity import check_bf16_output
from test_gpu_quantized_output import _check_oracle, _check_own_quantizer

import fp8_precision_recommendation_gb300 as loka

pytestmark = pytest.mark.gpu

DEV = "cuda"
BLK = W.NORM_BLOCK_RMS


def _gpu(t):
    return t.to(DEV) if t is not None else None


def _layer(inp, out_mode=None):
    return loka.Layer(x=_gpu(inp.x), w=_gpu(inp.w), bias=_gpu(inp.bias), gamma=_gpu(inp.gamma),
                      beta=_gpu(inp.beta), mode=inp.mode, norm=inp.norm, eps=inp.eps, norm_block=inp.norm_block,
                      act=inp.act, y_q_mode=out_mode)


def _run(layers):
    loka.fp8_linear_norm(layers)
    torch.cuda.synchronize()
    assert loka._loka.loka_device_status() == 0
    return layers


def _case(M, K, N, mode, norm, block, act, gamma, seed, x_dist="normal"):
    inp = W.make_layer(M, K, N, mode=mode, norm=norm, seed=seed, x_dist=x_dist, bias_var=0.02,
                       outlier_frac=0.01 if x_dist == "normal" else 0.0, gamma_uniform=gamma)
    inp.norm_block = block
    inp.act = act
    return inp


def _check(inp, layer, rows=None, what=""):
    y, _, _ = OL.linear_norm_inputs(inp, rows=rows)
    g = layer.y.cpu() if rows is None else layer.y[torch.as_tensor(rows)].cpu()
    check_bf16_output(g, y, normalized=inp.norm != W.NORM_NONE, what=what)


@pytest.mark.parametrize("block", [32, 64, 128, 256])
@pytest.mark.parametrize("N", [256, 512, 2048])
@pytest.mark.parametrize("act", [W.ACT_NONE, W.ACT_HARDSWISH])
def test_blocknorm_shapes(lib, block, N, act):
    # N > 256 splits rows over a cluster; BlockNorm needs no exchange there
    inp = _case(389, 256, N, W.SCALE_ROW, BLK, block, act, gamma=block != 64, seed=block + N + act)
    (layer,) = _run([_layer(inp)])
    _check(inp, layer, what=f"block{block} N{N} act{act}")


@pytest.mark.parametrize("N,block", [(64, 32), (64, 64), (192, 32), (192, 64), (128, 128)])
def test_blocknorm_narrow_rows(lib, N, block):
    inp = _case(300, 128, N, W.SCALE_ROW, BLK, block, W.ACT_HARDSWISH, gamma=True, seed=N * block)
    (layer,) = _run([_layer(inp)])
    _check(inp, layer, what=f"N{N} block{block}")


@pytest.mark.parametrize("norm", [W.NORM_NONE, W.NORM_LAYER, W.NORM_RMS])
@pytest.mark.parametrize("mode", [W.SCALE_TENSOR, W.SCALE_ROW, W.SCALE_MX32, W.SCALE_BF16])
def test_hard_swish_with_every_norm_and_scaling(lib, norm, mode):
    inp = _case(300, 256, 256, mode, norm, 256, W.ACT_HARDSWISH, gamma=True, seed=10 * norm + mode)
    inp.beta = W.random_bf16((256,), seed=3, var=0.1)
    (layer,) = _run([_layer(inp)])
    _check(inp, layer, what=f"hswish norm{norm} mode{mode}")


@pytest.mark.parametrize("mode", [W.SCALE_MX32, W.SCALE_BF16])
def test_blocknorm_mx_and_bf16_paths(lib, mode):
    inp = _case(500, 512, 1024, mode, BLK, 256, W.ACT_HARDSWISH, gamma=True, seed=30 + mode, x_dist="laplace")
    (layer,) = _run([_layer(inp)])
    _check(inp, layer, what=f"mode{mode}")


@pytest.mark.parametrize("out_mode,N,block", [(W.SCALE_ROW, 256, 64), (W.SCALE_ROW, 192, 32),
                                               (W.SCALE_MX32, 256, 128), (W.SCALE_MX32, 2048, 256)])
@pytest.mark.parametrize("act", [W.ACT_NONE, W.ACT_HARDSWISH])
def test_blocknorm_quantized_output(lib, out_mode, N, block, act):
    inp = _case(389, 256, N, W.SCALE_ROW, BLK, block, act, gamma=True, seed=50 + N + block + act)
    (layer,) = _run([_layer(inp, out_mode)])
    what = f"out{out_mode} N{N} block{block} act{act}"
    _check_own_quantizer(layer, out_mode, what)
    _check_oracle(inp, out_mode, layer, what=what)


@pytest.mark.parametrize("out_mode", [W.SCALE_ROW, W.SCALE_MX32])
@pytest.mark.parametrize("norm", [W.NORM_LAYER, W.NORM_RMS, W.NORM_NONE])
def test_hard_swish_quantized_output(lib, out_mode, norm):
    # Hard Swish is not monotone: the row amax comes from the amax pass
    inp = _case(389, 256, 256, W.SCALE_ROW, norm, 256, W.ACT_HARDSWISH, gamma=False, seed=70 + norm + out_mode)
    (layer,) = _run([_layer(inp, out_mode)])
    what = f"hswish out{out_mode} norm{norm}"
    _check_own_quantizer(layer, out_mode, what)
    _check_oracle(inp, out_mode, layer, what=what)


def test_blocknorm_grouped_ragged(lib):
    inps = [_case(m, 256, 512, W.SCALE_ROW, BLK, 128, W.ACT_HARDSWISH, gamma=True, seed=90 + m) for m in (300, 0, 129, 1)]
    layers = _run([_layer(i) for i in inps])
    for inp, layer in zip(inps, layers):
        if inp.M:
            _check(inp, layer, what=f"group M{inp.M}")


def test_blocknorm_wide_layer_full_size(lib):
    # a wide LRM layer: X [65536, 512], N = 2048, BlockNorm 256 + Hard Swish
    inp = _case(65536, 512, 2048, W.SCALE_ROW, BLK, 256, W.ACT_HARDSWISH, gamma=False, seed=0)
    (layer,) = _run([_layer(inp)])
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([np.arange(128), rng.integers(0, inp.M, 512), np.arange(inp.M - 128, inp.M)]))
    _check(inp, layer, rows=rows, what="wide blocknorm")
