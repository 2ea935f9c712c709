"""The channel-major tensor-core kernel (x in boxes of whole output rows or im2col boxes,
weights resident in tensor memory or loaded with every K step) against the oracle, every
element (GPU only).

Each case forces one variant through cbs_plan_request (row_boxes, weights_resident) on
shapes that reach its edges: the full-size downsample and pointwise layers; 16/32/64-
channel K steps; 3x3, 5x5, 2x2 and 1x1 filters; strides 1 and 2 (the stride-2 row boxes
read x as pixel pairs); one to four channel tiles with a ragged last one; a short last
row group; pixel counts that are not a multiple of 16 or of the unit (im2col units); a
share of a single 16-pixel chunk; and the run-time epilogue modes (identity, ReLU).
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import (LAYERS, LayerShape, bf16_bits_to_f32, bits_to_torch_bf16,
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


def _inputs(capi, shape, seed):
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=seed)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    return inp, x, w, scale, bias


def _check(got_t, ref, what):
    got = bf16_bits_to_f32(torch_bf16_to_bits(got_t)).astype(np.float64)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; worst at {idx}: "
                             f"gpu {got[idx]!r} oracle {ref[idx]!r}")


ROW_CASES = [
    # n, h, w, c, c_out, r, stride, pad
    (16, 160, 160, 64, 128, 3, 2, 1),   # the downsample layer: 3-row units, short last group
    (16, 40, 40, 256, 256, 1, 1, 0),    # the pointwise layer: 6-row units, two channel tiles
    (3, 32, 32, 16, 200, 3, 2, 1),      # 16-channel K steps, a ragged second channel tile
    (2, 24, 48, 64, 64, 3, 1, 1),       # stride 1, short last group
    (1, 32, 32, 128, 512, 1, 1, 0),     # four channel tiles
    (2, 33, 32, 96, 136, 1, 2, 0),      # 1x1 stride 2 on pixel pairs, 32-channel K steps
    (4, 20, 20, 64, 64, 5, 1, 2),       # 5x5, pad 2
    (2, 32, 32, 32, 64, 2, 2, 0),       # 2x2 stride 2 (patchify)
]

IM2COL_CASES = [
    (2, 17, 19, 32, 48, 3, 1, 1),       # 32-channel K steps, c_out below one tile
    (3, 9, 13, 16, 200, 3, 2, 1),       # 16-channel K steps, a ragged second channel tile
    (4, 21, 23, 64, 64, 3, 1, 1),       # pixel count not a multiple of 16
    (1, 4, 4, 64, 128, 3, 1, 1),        # 16 pixels: one chunk, most CTAs idle
]


def _run_variant(capi, case, **req):
    n, h, w, c, k, r, stride, pad = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = capi.plan_request(n, h, w, c, k, r, r, stride, pad, sms, **req)
    assert p["swap_ab"] == 1, p
    for key, val in req.items():
        assert p[key] == val, (key, p)
    shape = LayerShape("cmajor", n, h, w, c, k, r, r, stride, pad)
    inp, x, wt, scale, bias = _inputs(capi, shape, seed=700 + c + k)
    y = capi.forward_request(x, wt, scale, bias, stride, pad, **req)
    torch.cuda.synchronize()
    capi.check()
    ref = oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps,
                              stride, pad)
    _check(y, ref, f"{case} {req}")
    # Deterministic: a second run is bit-identical.
    y2 = capi.forward_request(x, wt, scale, bias, stride, pad, **req)
    torch.cuda.synchronize()
    assert np.array_equal(torch_bf16_to_bits(y), torch_bf16_to_bits(y2))


def _ids(cases):
    return [f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}-{c[5]}x{c[5]}s{c[6]}p{c[7]}" for c in cases]


@pytest.mark.parametrize("case", ROW_CASES, ids=_ids(ROW_CASES))
def test_row_boxes_streamed_weights(capi, case):
    _run_variant(capi, case, row_boxes=1, weights_resident=0)


@pytest.mark.parametrize("case", ROW_CASES[:3] + ROW_CASES[7:], ids=_ids(ROW_CASES[:3] + ROW_CASES[7:]))
def test_row_boxes_resident_weights(capi, case):
    _run_variant(capi, case, row_boxes=1, weights_resident=1)


@pytest.mark.parametrize("case", ROW_CASES[:1] + IM2COL_CASES, ids=_ids(ROW_CASES[:1] + IM2COL_CASES))
def test_im2col_boxes_resident_weights(capi, case):
    _run_variant(capi, case, row_boxes=0, weights_resident=1)


@pytest.mark.parametrize("activation", ["identity", "relu"])
def test_channel_major_other_activations(capi, activation):
    """The run-time epilogue modes on the kernel the planner picks for the downsample layer."""
    sh = LAYERS["down"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = capi.plan(sh.n, sh.h, sh.w, sh.c, sh.k, sh.r, sh.s, sh.stride, sh.pad, "auto", sms)
    assert p["row_boxes"] == 1, p
    inp, x, wt, scale, bias = _inputs(capi, sh, seed=711)
    y = capi.forward_act(x, wt, scale, bias, sh.stride, sh.pad, activation=activation)
    torch.cuda.synchronize()
    capi.check()
    ref = oracle.conv_bn_act(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps,
                             sh.stride, sh.pad, activation=activation)
    _check(y, ref, f"down ({activation}, row boxes)")


def test_x_modes_on_the_same_buffers(capi):
    """A 1x1 layer's matrix-row units and its im2col units, on the same x, w and y one after
    another: the two kinds of x tensor map have the same pixels per unit here, and each call
    must get its own kind (an im2col load issued with a tiled map is an illegal instruction)."""
    n, h, w, c, k = 2, 40, 40, 64, 64
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    matrix = capi.plan_request(n, h, w, c, k, 1, 1, 1, 0, sms, row_boxes=1, weights_resident=1)
    im2col = capi.plan_request(n, h, w, c, k, 1, 1, 1, 0, sms, row_boxes=0, weights_resident=1)
    assert matrix["row_boxes"] == 1 and im2col["row_boxes"] == 0
    assert matrix["block_m"] == im2col["block_m"], (matrix, im2col)  # same pixels per unit
    shape = LayerShape("modes", n, h, w, c, k, 1, 1, 1, 0)
    inp, x, wt, scale, bias = _inputs(capi, shape, seed=733)
    ref = oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps, 1, 0)
    y = torch.empty((n, h, w, k), dtype=torch.bfloat16, device=x.device)
    order = [{"row_boxes": 1, "weights_resident": 1}, {"row_boxes": 0, "weights_resident": 1},
             {"row_boxes": 1, "weights_resident": 0}, {"row_boxes": 0, "weights_resident": 1}, {}]
    for req in order:
        y.fill_(float("nan"))
        capi.forward_request(x, wt, scale, bias, 1, 0, y=y, **req)
        torch.cuda.synchronize()
        capi.check()
        _check(y, ref, f"x mode {req}")
