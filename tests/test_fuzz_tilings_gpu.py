"""Seeded random layer shapes, every tiling each admits (GPU only).

For each shape drawn from a fixed seed (batch, odd and even sizes, 16-128 input
channels, 8-264 output channels, 1x1/3x3/5x5 filters, stride 1 or 2, zero or
"same" padding), the planner's choice and every tcgen05 alternative that
conv_bn_silu_plan_request accepts for it (pixel-major 128/256-wide tiles,
stream-K, 2-CTA pairs, channel-major whole tiles and balanced runs) and the
direct kernel run through conv_bn_silu_forward_request; every output element is
compared with the fp64 oracle at the layer's tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import (LayerShape, bf16_bits_to_f32, bits_to_torch_bf16,
                                                   make_layer_inputs, torch_bf16_to_bits)

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


def random_shapes(count: int, seed: int = 20261202):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        r = int(rng.choice([1, 3, 3, 5]))
        stride = int(rng.choice([1, 2]))
        pad = int(rng.choice([0, r // 2]))
        n = int(rng.integers(1, 4))
        h, w = (int(v) for v in rng.integers(1, 49, size=2))
        c = int(rng.choice([16, 32, 48, 64, 96, 128]))
        k = int(rng.choice([8, 16, 24, 40, 64, 72, 128, 136, 200, 256, 264]))
        if (h + 2 * pad - r) < 0 or (w + 2 * pad - r) < 0:
            continue
        out.append(LayerShape(f"fz{len(out)}", n, h, w, c, k, r, r, stride, pad))
    return out


SHAPES = random_shapes(14)


def _variants():
    from conv2d_batchnorm_silu_gb300 import tune
    return list(tune.variants())


@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s.n}x{s.h}x{s.w}x{s.c}-{s.k}-r{s.r}s{s.stride}p{s.pad}"
                                               for s in SHAPES])
def test_every_admitted_tiling_matches_oracle(capi, shape):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=shape.h * 131 + shape.w)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    ref = oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps,
                              shape.stride, shape.pad)
    ran = []
    for label, ov in _variants():
        try:
            capi.plan_request(shape.n, shape.h, shape.w, shape.c, shape.k, shape.r, shape.s, shape.stride,
                              shape.pad, sms, **ov)
        except capi.CbsError:
            continue
        y = capi.forward_request(x, w, scale, bias, shape.stride, shape.pad, **ov)
        torch.cuda.synchronize()
        capi.check()
        got = bf16_bits_to_f32(torch_bf16_to_bits(y)).astype(np.float64)
        err = np.abs(got - ref)
        bound = ATOL + RTOL * np.abs(ref)
        assert np.all(np.isfinite(got)), (label, "non-finite output")
        assert np.all(err <= bound), (label, int((err > bound).sum()), float((err - bound).max()))
        ran.append(label)
    assert "auto" in ran and "direct" in ran, ran
