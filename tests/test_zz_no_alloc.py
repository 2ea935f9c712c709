"""The allocation-free forward entry point (GPU only).

conv_bn_silu_forward_noalloc serves callers that may not allocate device
memory (a framework's caching allocator owns it all, a fixed memory budget, a
loop that cannot afford cudaMalloc's synchronisation).  It must give the same
result as conv_bn_silu_forward, within the layer's bf16 tolerance, call after
call, while its stream-K scratch lives in one fixed device array that every
call reuses.  This file is named to be collected last; it also passes when
run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from conv2d_batchnorm_silu_gb300.synthetic import (LAYERS, LayerShape, bf16_bits_to_f32,
                                                   bits_to_torch_bf16, make_layer_inputs,
                                                   torch_bf16_to_bits)

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="module")
def capi():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from conv2d_batchnorm_silu_gb300 import _build
    _build.build()
    from conv2d_batchnorm_silu_gb300 import capi as c
    return c


def _device_inputs(capi, shape, seed):
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=seed)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    return x, w, scale, bias


def _f64(y):
    return bf16_bits_to_f32(torch_bf16_to_bits(y)).astype(np.float64)


SHAPES = [
    LAYERS["deep"],                                                 # stream-K, 200 tiles
    LayerShape("split244", 39, 20, 20, 256, 384, 3, 3, 1, 1),       # stream-K, ragged tails
    LAYERS["down"],                                                 # whole tiles, no scratch
]


@pytest.mark.parametrize("shape", SHAPES, ids=[s.name for s in SHAPES])
def test_noalloc_matches_forward_on_two_calls_in_a_row(capi, shape):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = capi.plan(shape.n, shape.h, shape.w, shape.c, shape.k, shape.r, shape.s,
                     shape.stride, shape.pad, "auto", sms)
    if shape.name != "down":
        assert plan["stream_k"] == 1, plan   # the scratch array is really used
    for seed in (101, 202):                  # two calls in a row, different data
        x, w, scale, bias = _device_inputs(capi, shape, seed)
        y_ref = capi.forward(x, w, scale, bias, shape.stride, shape.pad)
        y = torch.full_like(y_ref, float("nan"))
        capi.forward_noalloc(x, w, scale, bias, y, shape.stride, shape.pad)
        torch.cuda.synchronize()
        capi.check()
        ref = _f64(y_ref)
        got = _f64(y)
        assert np.all(np.isfinite(got))
        err = np.abs(got - ref)
        assert np.all(err <= ATOL + RTOL * np.abs(ref)), (shape.name, seed, float(err.max()))
