"""Other epilogues on the GPU (conv_bn_act_forward): identity and ReLU after the
BN multiply/add, and a residual added after the activation ("Fusing an
Epilogue", section "What an epilogue is").  Every kernel family is exercised
-- the tcgen05 kernel in its pixel-major, channel-major (swap) and 2-CTA
stream-K forms, the thin-input kernel and the CUDA-core direct kernel -- and
every output element is compared with the fp64 oracle at the layer's
tolerance |err| <= 1e-2 + 1e-2*|ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import (LayerShape, bf16_bits_to_f32, bits_to_torch_bf16,
                                                   f32_to_bf16_bits, make_layer_inputs, torch_bf16_to_bits)

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


SHAPES = [
    (LayerShape("tiny", 1, 32, 32, 16, 32, 3, 3, 1, 1), "tcgen05 pixel-major"),
    (LayerShape("ragged", 2, 13, 11, 16, 24, 3, 3, 1, 1), "tcgen05 pixel-major, channel tail"),
    (LayerShape("swap", 2, 100, 100, 16, 80, 3, 3, 1, 1), "tcgen05 channel-major (swap AB)"),
    (LayerShape("pairs", 31, 20, 20, 128, 512, 3, 3, 1, 1), "tcgen05 2-CTA stream-K"),
    (LayerShape("c2f", 8, 80, 80, 128, 128, 1, 1, 1, 0), "tcgen05 channel-major, balanced runs"),
    (LayerShape("thin", 1, 64, 64, 3, 16, 3, 3, 2, 1), "thin-input tcgen05"),
    (LayerShape("direct", 1, 9, 7, 5, 12, 3, 3, 2, 1), "CUDA-core direct"),
]
CASES = [(sh, what, act, res) for sh, what in SHAPES for act in ("identity", "relu", "silu")
         for res in (False, True)]


def _f64(t):
    return bf16_bits_to_f32(torch_bf16_to_bits(t)).astype(np.float64)


def _check(got, ref, what):
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; worst at {i}: "
                             f"gpu {got[i]!r} oracle {ref[i]!r}")


def _run(capi, shape, activation, with_residual, seed, in_place=False):
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=seed)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    out_shape = (shape.n, shape.ho, shape.wo, shape.k)
    res_bits = None
    res = None
    if with_residual:
        rng = np.random.default_rng(seed + 1)
        res_bits = f32_to_bf16_bits(rng.standard_normal(out_shape).astype(np.float32))
        res = bits_to_torch_bf16(res_bits).to(dev)
    y = res if in_place else None
    y = capi.forward_act(x, w, scale, bias, shape.stride, shape.pad, activation=activation, residual=res, y=y)
    torch.cuda.synchronize()
    capi.check()
    ref = oracle.conv_bn_act(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps,
                             shape.stride, shape.pad, activation, res_bits)
    return _f64(y), ref


@pytest.mark.parametrize("shape,what,activation,with_residual", CASES,
                         ids=[f"{c[0].name}-{c[2]}-{'res' if c[3] else 'nores'}" for c in CASES])
def test_epilogue_matches_oracle(capi, shape, what, activation, with_residual):
    got, ref = _run(capi, shape, activation, with_residual, seed=77)
    _check(got, ref, f"{shape.name} ({what}) {activation} residual={with_residual}")


@pytest.mark.parametrize("name", ["tiny", "swap", "pairs", "c2f", "thin", "direct"])
def test_residual_in_place(capi, name):
    """residual == y: each element's residual is read before its result is stored."""
    shape = next(s for s, _ in SHAPES if s.name == name)
    got, ref = _run(capi, shape, "silu", True, seed=91, in_place=True)
    _check(got, ref, f"{name} in place")


def test_silu_without_residual_is_bit_identical_to_the_layer(capi):
    shape = SHAPES[2][0]
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=5)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    a = capi.forward(x, w, scale, bias, shape.stride, shape.pad)
    c = capi.forward_act(x, w, scale, bias, shape.stride, shape.pad, activation="silu")
    torch.cuda.synchronize()
    assert torch.equal(a, c)
