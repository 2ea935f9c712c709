"""The allocation-free forward entry point (GPU only).

conv_bn_silu_forward_noalloc serves callers that may not allocate device
memory (a framework's caching allocator owns it all, a fixed memory budget, a
loop that cannot afford cudaMalloc's synchronisation).  It runs the same plan
as conv_bn_silu_forward, so its output must be bit-identical to that entry
point's, and every element must match the oracle within the layer's bf16
tolerance, call after call, while its stream-K scratch lives in one fixed
device array that every call reuses.  The calls under test must also leave the
device's free memory unchanged.  This file is named to be collected last; it
also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import (LAYERS, LayerShape, bf16_bits_to_f32,
                                                   bits_to_torch_bf16, make_layer_inputs,
                                                   torch_bf16_to_bits)

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
SEEDS = (101, 202)   # two calls in a row per shape, on different data


@pytest.fixture(scope="module")
def capi():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from conv2d_batchnorm_silu_gb300 import _build
    _build.build()
    from conv2d_batchnorm_silu_gb300 import capi as c
    return c


def _device_inputs(capi, inp):
    dev = torch.device("cuda:0")
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    return x, w, scale, bias


def _bits(y):
    return torch_bf16_to_bits(y)


SHAPES = [
    LAYERS["deep"],                                                 # stream-K pairs, 100 pair tiles
    LayerShape("split244", 39, 20, 20, 256, 384, 3, 3, 1, 1),       # stream-K, ragged tails
    LAYERS["down"],                                                 # whole tiles, no scratch
]


def test_noalloc_bit_identical_to_forward_and_matches_oracle(capi):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for sh in SHAPES:
        p = capi.plan(sh.n, sh.h, sh.w, sh.c, sh.k, sh.r, sh.s, sh.stride, sh.pad, "auto", sms)
        if sh.name != "down":
            assert p["stream_k"] == 1, (sh.name, p)     # the scratch array is really used

    # Every tensor is allocated, and every kernel the calls need is loaded, before the
    # free-memory reading: the regular entry point runs each shape once on the default
    # stream, and the allocation-free one runs its per-device set-up on a small layer.
    cases = []
    for sh in SHAPES:
        for seed in SEEDS:
            inp = make_layer_inputs(sh, seed=seed)
            x, w, scale, bias = _device_inputs(capi, inp)
            y = torch.full((sh.n, sh.ho, sh.wo, sh.k), float("nan"), dtype=torch.bfloat16,
                           device="cuda:0")
            cases.append((sh, inp, x, w, scale, bias, y))
    for sh, _, x, w, scale, bias, _ in cases[::len(SEEDS)]:
        capi.forward(x, w, scale, bias, sh.stride, sh.pad)
    tiny = LAYERS["tiny"]
    tx, tw, ts, tb = _device_inputs(capi, make_layer_inputs(tiny))
    ty = torch.empty((tiny.n, tiny.ho, tiny.wo, tiny.k), dtype=torch.bfloat16, device="cuda:0")
    capi.forward_noalloc(tx, tw, ts, tb, ty, tiny.stride, tiny.pad)
    torch.cuda.synchronize()
    capi.check()

    # The calls under test run on a stream the library has never seen: a call that fell
    # back to the library-held stream-K workspace would allocate one for it.
    stream = torch.cuda.Stream()
    free_before, _ = torch.cuda.mem_get_info()
    for sh, _, x, w, scale, bias, y in cases:
        capi.forward_noalloc(x, w, scale, bias, y, sh.stride, sh.pad, stream=stream)
    stream.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    capi.check(stream)
    assert free_after == free_before, ("the allocation-free calls changed free device memory",
                                       free_before, free_after)

    for sh, inp, x, w, scale, bias, y in cases:
        y_ref = capi.forward(x, w, scale, bias, sh.stride, sh.pad)
        torch.cuda.synchronize()
        capi.check()
        assert np.array_equal(_bits(y), _bits(y_ref)), f"{sh.name}: not bit-identical to conv_bn_silu_forward"
        got = bf16_bits_to_f32(_bits(y)).astype(np.float64)
        ref = oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var,
                                  inp.eps, sh.stride, sh.pad)
        assert np.all(np.isfinite(got)), sh.name
        err = np.abs(got - ref)
        bound = ATOL + RTOL * np.abs(ref)
        assert np.all(err <= bound), (sh.name, float((err - bound).max()))
