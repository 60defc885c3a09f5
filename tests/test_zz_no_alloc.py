"""The allocation-free entry point loka_fp8_linear_norm_static.

It serves callers that cannot allocate device memory and so cannot pass the
workspace loka_fp8_linear_norm needs: it uses the library's built-in 4 MiB
scratch array instead.  Checked through the C ABI against the workspace
entry point on the same inputs, on two calls in a row (the array keeps the
previous call's contents, so the second call must clear what it needs)."""
import pytest
import torch

import workloads as W
import fp8_precision_recommendation_gb300 as loka
from fp8_precision_recommendation_gb300 import _loka

pytestmark = pytest.mark.gpu


def _layers(inp, dev):
    def mk():
        return loka.Layer(x=inp.x.to(dev), w=inp.w.to(dev), bias=None if inp.bias is None else inp.bias.to(dev),
                          gamma=None if inp.gamma is None else inp.gamma.to(dev), mode=inp.mode, norm=inp.norm,
                          eps=inp.eps)
    return mk


@pytest.mark.parametrize("mode,norm,K,N", [(W.SCALE_ROW, W.NORM_LAYER, 512, 256), (W.SCALE_TENSOR, W.NORM_RMS, 512, 256),
                                           (W.SCALE_ROW, W.NORM_LAYER, 96, 160), (W.SCALE_MX32, W.NORM_RMS, 64, 320)])
def test_static_scratch_matches_workspace_entry_point_twice(lib, mode, norm, K, N):
    dev = torch.device("cuda")
    inp = W.make_layer(2000, K, N, mode=mode, norm=norm, seed=41, bias_var=0.02, outlier_frac=0.01,
                       gamma_uniform=True)
    mk = _layers(inp, dev)
    ref = mk()
    (y_ref,) = loka.fp8_linear_norm([ref])
    for call in range(2):
        layer = mk()
        d = layer.desc()
        layer.y.fill_(float("nan"))
        _loka.loka_fp8_linear_norm_static([d])
        torch.cuda.synchronize()
        assert _loka.loka_device_status() == _loka.LOKA_OK
        diff = (layer.y.float() - y_ref.float()).abs().max().item()
        assert diff == 0.0, f"call {call}: max difference {diff}"


def test_static_scratch_rejects_too_large_problems(lib):
    dev = torch.device("cuda")
    # tensorwise scaling quantizes X into scratch first: 8 MiB of E4M3
    # activations > 4 MiB
    M, K, N = 16384, 512, 256
    layer = loka.Layer(x=torch.zeros((M, K), dtype=torch.bfloat16, device=dev),
                       w=torch.zeros((N, K), dtype=torch.bfloat16, device=dev), mode=W.SCALE_TENSOR,
                       norm=W.NORM_LAYER, eps=1e-5)
    with pytest.raises(_loka.LokaError) as e:
        _loka.loka_fp8_linear_norm_static([layer.desc()])
    assert e.value.status == _loka.LOKA_ERR_WORKSPACE


@pytest.mark.parametrize("out_mode", [W.SCALE_ROW, W.SCALE_MX32])
def test_static_scratch_quantized_output(lib, out_mode):
    # the E4M3 output for the next layer through the allocation-free call:
    # the same codes and scales as through the workspace entry point
    dev = torch.device("cuda")
    inp = W.make_layer(1500, 512, 256, mode=W.SCALE_ROW, norm=W.NORM_LAYER, seed=43, bias_var=0.02)
    mk = _layers(inp, dev)
    ref = mk()
    ref.y_q_mode = out_mode
    loka.fp8_linear_norm([ref])
    layer = mk()
    layer.y_q_mode = out_mode
    layer.y_q_only = True
    d = layer.desc()
    layer.y_q.fill_(0xFF)
    _loka.loka_fp8_linear_norm_static([d])
    torch.cuda.synchronize()
    assert _loka.loka_device_status() == _loka.LOKA_OK
    assert torch.equal(layer.y_q, ref.y_q)
    assert torch.equal(layer.y_q_scales, ref.y_q_scales)
