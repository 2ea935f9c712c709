"""The unfused comparator (GPU only): conv -> t1, BN -> t2, SiLU -> y as three
kernels, the sequence the fusion replaces ("Fusing an Epilogue", kernels
book, section "The problem").

Each step is checked against the oracle on its own seeded input, with a bound
derived from the rounding the step performs:

* conv (the forward kernel reduced to the bf16 cast): |t1 - acc| <= 2^-8 |acc|
  for the bf16 rounding, plus 2e-3 + 1e-3 |acc| for fp32 accumulation order;
* BN alone: t2 = bf16(fp32(t1*scale + bias)), |t2 - z| <= 2^-8 |z| (1 + 2^-10);
* SiLU alone: |y - SiLU(t2)| <= 2^-8 |SiLU(t2)| + 2e-5 (bf16 rounding plus the
  hardware tanh's error, below 1e-5 on the real line);
* t2 inside the sequence: BN of the rounded t1, rounded once more;
* the whole sequence against the fp64 layer: the layer tolerance
  1e-2 + 1e-2 |y| plus what the two intermediate roundings can move z by,
  |scale * acc| 2^-8 + |z| 2^-8, times 1.1 (SiLU's slope is at most 1.0999).
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import (LAYERS, LayerShape, bf16_bits_to_f32,
                                                   bits_to_torch_bf16, f32_to_bf16_bits,
                                                   make_layer_inputs, torch_bf16_to_bits)

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
U = 2.0 ** -8          # bf16 round-to-nearest: relative error at most half of 2^-7
SILU_SLOPE = 1.1       # max |d/dz z*sigmoid(z)| = 1.0998...


@pytest.fixture(scope="module")
def capi():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from conv2d_batchnorm_silu_gb300 import _build
    _build.build()
    from conv2d_batchnorm_silu_gb300 import capi as c
    return c


def f64(t):
    return bf16_bits_to_f32(torch_bf16_to_bits(t)).astype(np.float64)


def check(got, ref, bound, what):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of bound; worst at {i}: "
                             f"gpu {got[i]!r} oracle {ref[i]!r} bound {bound[i]!r}")


def device_layer(capi, inp):
    dev = torch.device("cuda:0")
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    return x, w, scale, bias


def unfused_bounds(acc, scale, bias):
    """Oracle z and y with the sequence's tolerance (see the module docstring)."""
    z = oracle.bn(acc, scale, bias)
    y = oracle.silu(z)
    drift = SILU_SLOPE * U * (np.abs(acc * scale) + np.abs(z))
    return y, ATOL + RTOL * np.abs(y) + drift


SMALL = [
    LAYERS["tiny"],
    LAYERS["stem"],                                               # thin-input kernel
    LAYERS["pointwise"],                                          # swap-AB
    LayerShape("odd", 2, 13, 11, 16, 24, 3, 3, 1, 1),             # ragged tiles
    LayerShape("direct", 1, 9, 7, 5, 12, 3, 3, 2, 1),             # direct kernel, c_out % 8 != 0
    LayerShape("splitk", 2, 10, 10, 256, 384, 3, 3, 1, 1),        # stream-K combine
]


@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_unfused_sequence_full(capi, shape):
    inp = make_layer_inputs(shape, seed=4242)
    x, w, scale, bias = device_layer(capi, inp)
    y, t1, t2 = capi.forward_unfused(x, w, scale, bias, shape.stride, shape.pad)
    torch.cuda.synchronize()
    capi.check()
    acc = oracle.conv2d(inp.x_bits, inp.w_bits, shape.stride, shape.pad)
    check(f64(t1), acc, U * np.abs(acc) + 2e-3 + 1e-3 * np.abs(acc), f"{shape.name} t1")
    sc = scale.cpu().numpy().astype(np.float64)
    bi = bias.cpu().numpy().astype(np.float64)
    y_ref, bound = unfused_bounds(acc, sc, bi)
    check(f64(y), y_ref, bound, f"{shape.name} y")
    # t2 is BN of the rounded t1, rounded once more
    z = oracle.bn(acc, sc, bi)
    t1_err = U * np.abs(acc) + 2e-3 + 1e-3 * np.abs(acc)
    check(f64(t2), z, np.abs(sc) * t1_err * (1 + U) + U * (1 + U) * np.abs(z) + 1e-6, f"{shape.name} t2")


@pytest.mark.parametrize("name", ["down", "deep"])
def test_unfused_sequence_sampled(capi, name):
    shape = LAYERS[name]
    inp = make_layer_inputs(shape)
    x, w, scale, bias = device_layer(capi, inp)
    y, t1, _ = capi.forward_unfused(x, w, scale, bias, shape.stride, shape.pad)
    torch.cuda.synchronize()
    capi.check()
    rng = np.random.default_rng(23)
    pix = np.unique(np.concatenate([rng.choice(shape.m, 2000, replace=False), [0, shape.m - 1]]))
    acc = oracle.conv2d_at(inp.x_bits, inp.w_bits, pix, shape.stride, shape.pad)
    t1s = f64(t1).reshape(-1, shape.k)[pix]
    check(t1s, acc, U * np.abs(acc) + 2e-3 + 1e-3 * np.abs(acc), f"{name} t1 (sampled)")
    y_ref, bound = unfused_bounds(acc, scale.cpu().numpy().astype(np.float64),
                                  bias.cpu().numpy().astype(np.float64))
    check(f64(y).reshape(-1, shape.k)[pix], y_ref, bound, f"{name} y (sampled)")


@pytest.mark.parametrize("c_out,count", [(128, 128 * 1000), (24, 24 * 333), (5, 5 * 77), (16, 0)])
def test_bn_apply_step(capi, c_out, count):
    """The BN kernel alone on seeded bf16 input: vector path (c_out % 8 == 0) and scalar path."""
    rng = np.random.default_rng(c_out * 7 + count)
    t1_bits = f32_to_bf16_bits(rng.normal(0, 3, count).astype(np.float32))
    g = rng.uniform(0.5, 1.5, c_out).astype(np.float32)
    b = rng.normal(0, 0.1, c_out).astype(np.float32)
    m = rng.normal(0, 0.1, c_out).astype(np.float32)
    v = rng.uniform(0.5, 2, c_out).astype(np.float32)
    sc64, bi64 = oracle.bn_fold(g, b, m, v, np.float32(1e-3))
    sc32, bi32 = sc64.astype(np.float32), bi64.astype(np.float32)   # what the kernel receives
    dev = torch.device("cuda:0")
    t1 = bits_to_torch_bf16(t1_bits).to(dev).reshape(-1, c_out)
    t2 = capi.bn_apply(t1, torch.from_numpy(sc32).to(dev), torch.from_numpy(bi32).to(dev))
    torch.cuda.synchronize()
    if count == 0:
        return
    z = oracle.bn(bf16_bits_to_f32(t1_bits).astype(np.float64).reshape(-1, c_out),
                  sc32.astype(np.float64), bi32.astype(np.float64))
    check(f64(t2), z, U * np.abs(z) * (1 + 2.0 ** -10) + 1e-37, f"bn_apply c_out={c_out}")


@pytest.mark.parametrize("count", [8 * 40000, 8 * 3 + 5])
def test_silu_apply_step(capi, count):
    """The SiLU kernel alone, over a spread of z including both tails and zero."""
    rng = np.random.default_rng(count)
    z = np.concatenate([rng.normal(0, 4, count - 5), [0.0, -0.0, 30.0, -30.0, -100.0]])
    z_bits = f32_to_bf16_bits(z.astype(np.float32))
    dev = torch.device("cuda:0")
    y = capi.silu_apply(bits_to_torch_bf16(z_bits).to(dev))
    torch.cuda.synchronize()
    ref = oracle.silu(bf16_bits_to_f32(z_bits).astype(np.float64))
    check(f64(y), ref, U * np.abs(ref) + 2e-5, f"silu_apply count={count}")

