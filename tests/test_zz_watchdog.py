"""The bounded-wait watchdog on the GPU, made to fire on purpose.

Every pipeline wait of the tcgen05 kernel is bounded; a kernel whose wait runs
out records it, stops, waits for its own copies in flight, frees its tensor
memory and returns, and conv_bn_silu_check reports CBS_ERR_TIMEOUT.  A bound
of one nanosecond (cbs_plan_request.wait_timeout_ns) makes the waits run out
without any fault: nothing traps, nothing hangs.  After it, the same context
must run the layer correctly again (stream-K flags and tickets re-zeroed).
Named to be collected last; it also passes run alone.
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import (LayerShape, bf16_bits_to_f32, bits_to_torch_bf16,
                                                   make_layer_inputs, torch_bf16_to_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from conv2d_batchnorm_silu_gb300 import _build
    _build.build()
    from conv2d_batchnorm_silu_gb300 import capi as c
    return c


SHAPES = [
    LayerShape("single", 2, 40, 40, 64, 64, 3, 3, 1, 1),        # whole tiles, single CTAs
    LayerShape("pairs", 31, 20, 20, 128, 512, 3, 3, 1, 1),      # stream-K over 2-CTA pairs
    LayerShape("swap", 2, 100, 100, 16, 80, 3, 3, 1, 1),        # channel-major tiles
]


@pytest.mark.parametrize("shape", SHAPES, ids=[s.name for s in SHAPES])
def test_wait_runs_out_then_the_layer_runs_normally(capi, shape):
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=13)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    torch.cuda.synchronize()
    fired = 0
    for _ in range(3):
        capi.forward_request(x, w, scale, bias, shape.stride, shape.pad, wait_timeout_ns=1)
        torch.cuda.synchronize()       # the kernel returned: no hang, no fault
        try:
            capi.check()
        except capi.CbsError as e:
            assert e.status == capi.CBS_ERR_TIMEOUT, e
            fired += 1
    assert fired >= 1, "a 1 ns bound never ran out"
    capi.check()                       # the error word was cleared by the reporting check
    y = capi.forward(x, w, scale, bias, shape.stride, shape.pad)
    torch.cuda.synchronize()
    capi.check()
    got = bf16_bits_to_f32(torch_bf16_to_bits(y)).astype(np.float64)
    ref = oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps,
                              shape.stride, shape.pad)
    assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))
