"""Tilings forced through conv_bn_silu_forward_request (GPU only): every
alternative the planner can be overridden into must compute the same layer.
Each case runs a tcgen05 tiling the planner would not pick for that shape and
compares every output element with the fp64 oracle at the layer's tolerance.
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


CASES = [
    ("pairs_off", LayerShape("sk", 31, 20, 20, 128, 512, 3, 3, 1, 1), {"pair": 0}),
    ("streamk_off", LayerShape("sk", 31, 20, 20, 128, 512, 3, 3, 1, 1), {"stream_k": 0}),
    ("n128_whole", LayerShape("sk", 31, 20, 20, 128, 512, 3, 3, 1, 1), {"stream_k": 0, "block_n": 128}),
    ("n128_streamk", LayerShape("sk", 31, 20, 20, 128, 512, 3, 3, 1, 1), {"stream_k": 1, "block_n": 128}),
    ("swap_off_tail", LayerShape("sw", 2, 100, 100, 16, 80, 3, 3, 1, 1), {"swap_ab": 0}),
    ("pw_n256", LayerShape("pw", 16, 40, 40, 256, 256, 1, 1, 1, 0), {"swap_ab": 0, "block_n": 256}),
    ("pw_n64", LayerShape("pw", 4, 40, 40, 256, 256, 1, 1, 1, 0), {"swap_ab": 0, "block_n": 64}),
    ("swap_small", LayerShape("ss", 2, 13, 11, 16, 24, 3, 3, 1, 1), {"swap_ab": 1}),
    ("swap_small_tiles", LayerShape("ss", 2, 13, 11, 16, 24, 3, 3, 1, 1), {"swap_ab": 1, "balanced": 0}),
    # balanced runs crossing from the first channel tile into a partial second one
    ("swap_two_ctiles", LayerShape("bx", 3, 30, 30, 32, 200, 1, 1, 1, 0), {"swap_ab": 1}),
    # two balanced units per CTA (256 pixels and a remainder), a ragged last chunk
    ("swap_multi_unit_tail", LayerShape("bl", 3, 150, 151, 16, 40, 3, 3, 1, 1), {"balanced": 1}),
    ("pw_swap_tiles", LayerShape("pw", 4, 40, 40, 256, 256, 1, 1, 1, 0), {"swap_ab": 1, "balanced": 0}),
    ("direct", LayerShape("dd", 2, 13, 11, 16, 24, 3, 3, 1, 1), {"algo": "direct"}),
]


@pytest.mark.parametrize("name,shape,overrides", CASES, ids=[c[0] for c in CASES])
def test_forced_tiling_matches_oracle(capi, name, shape, overrides):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    forced = capi.plan_request(shape.n, shape.h, shape.w, shape.c, shape.k, shape.r, shape.s, shape.stride,
                               shape.pad, sms, **overrides)
    auto = capi.plan(shape.n, shape.h, shape.w, shape.c, shape.k, shape.r, shape.s, shape.stride, shape.pad,
                     "auto", sms)
    assert forced != auto, "the override must change the plan"
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=61)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    y = capi.forward_request(x, w, scale, bias, shape.stride, shape.pad, **overrides)
    torch.cuda.synchronize()
    capi.check()
    got = bf16_bits_to_f32(torch_bf16_to_bits(y)).astype(np.float64)
    ref = oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps,
                              shape.stride, shape.pad)
    err = np.abs(got - ref)
    bound = 1e-2 + 1e-2 * np.abs(ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= bound), (name, float((err - bound).max()))


@pytest.mark.parametrize("shape", [LayerShape("pointwise", 16, 40, 40, 256, 256, 1, 1, 1, 0),
                                   LayerShape("down", 16, 160, 160, 64, 128, 3, 3, 2, 1)],
                         ids=["pointwise", "down"])
def test_balanced_runs_equal_whole_tiles_bitwise(capi, shape):
    """Balanced runs and whole tiles cut the pixels differently but sum every output's K
    steps in the same order: the two schedules give bit-identical outputs."""
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=67)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    y1 = capi.forward_request(x, w, scale, bias, shape.stride, shape.pad, swap_ab=1, balanced=1)
    y0 = capi.forward_request(x, w, scale, bias, shape.stride, shape.pad, swap_ab=1, balanced=0)
    torch.cuda.synchronize()
    capi.check()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


def test_stream_k_plans_of_different_layouts_share_one_workspace(capi):
    """The library-held stream-K buffer serves plans of different layouts (2-CTA pairs,
    single CTAs, 128- and 256-channel tiles: different slot counts and partial-tile sizes)
    one after another on one stream: no plan's partial sums may land in another plan's
    flags, and the flags each plan leaves behind are zero."""
    shape = LayerShape("sk", 31, 20, 20, 128, 512, 3, 3, 1, 1)
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=83)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    ref = oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps,
                              shape.stride, shape.pad)
    bound = 1e-2 + 1e-2 * np.abs(ref)
    order = [{}, {"stream_k": 1, "block_n": 128}, {"pair": 0}, {"stream_k": 1, "block_n": 64}, {}]
    for ov in order * 2:
        y = capi.forward_request(x, w, scale, bias, shape.stride, shape.pad, **ov)
        torch.cuda.synchronize()
        capi.check()
        got = bf16_bits_to_f32(torch_bf16_to_bits(y)).astype(np.float64)
        assert np.all(np.abs(got - ref) <= bound), ov


MULTI_TILE_CASES = [
    # Several pixel tiles per CTA, and tiles whose epilogue warps hold chunks past the last
    # output channel next to live ones: such a chunk is neither staged nor stored, and the
    # staging buffers of the live chunks (reused by the CTA's next tile) stay consistent.
    ("n256_cout64", LayerShape("mt", 4, 160, 160, 16, 64, 3, 3, 1, 1),
     {"swap_ab": 0, "stream_k": 0, "pair": 0, "block_n": 256}),
    ("n128_cout80", LayerShape("mt", 4, 160, 160, 16, 80, 3, 3, 1, 1),
     {"swap_ab": 0, "stream_k": 0, "pair": 0, "block_n": 128}),
    ("n256_sk_cout64", LayerShape("mt", 4, 160, 160, 16, 64, 3, 3, 1, 1),
     {"swap_ab": 0, "stream_k": 1, "pair": 0, "block_n": 256}),
    # stream-K with tiles narrower than 128 channels: the combining piece's prefetch of its
    # partner's partial sums covers only the warp's own 32 or 16 accumulator columns
    ("n64_sk", LayerShape("mt", 4, 80, 80, 128, 64, 3, 3, 1, 1),
     {"swap_ab": 0, "stream_k": 1, "pair": 0, "block_n": 64}),
    ("n32_sk_ragged", LayerShape("mt", 4, 80, 80, 128, 48, 3, 3, 1, 1),
     {"swap_ab": 0, "stream_k": 1, "pair": 0, "block_n": 32}),
    ("swap_tiles_ragged", LayerShape("mt", 3, 100, 100, 64, 200, 3, 3, 1, 1), {"swap_ab": 1, "balanced": 0}),
]


@pytest.mark.parametrize("name,shape,overrides", MULTI_TILE_CASES, ids=[c[0] for c in MULTI_TILE_CASES])
def test_multi_tile_ctas_match_oracle(capi, name, shape, overrides):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = capi.plan_request(shape.n, shape.h, shape.w, shape.c, shape.k, shape.r, shape.s, shape.stride,
                             shape.pad, sms, **overrides)
    assert plan["tiles"] > plan["grid"], plan  # some CTA runs more than one tile
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=89)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    ref = oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps,
                              shape.stride, shape.pad)
    bound = 1e-2 + 1e-2 * np.abs(ref)
    y = torch.empty(ref.shape, dtype=torch.bfloat16, device=dev)
    for rep in range(3):  # a race shows on some runs only
        y.fill_(float("nan"))
        capi.forward_request(x, w, scale, bias, shape.stride, shape.pad, y=y, **overrides)
        torch.cuda.synchronize()
        capi.check()
        got = bf16_bits_to_f32(torch_bf16_to_bits(y)).astype(np.float64)
        err = np.abs(got - ref)
        assert np.all(np.isfinite(got)), (name, rep)
        assert np.all(err <= bound), (name, rep, int((err > bound).sum()), float((err - bound).max()))
