"""Pins for the oracle's BN fold, its SiLU and the whole composed layer (CPU only).

"Fusing an Epilogue", sections "The problem" and "The shape of it": batch
norm is a per-channel multiply and add on the convolution's result, and
SiLU multiplies a value by its sigmoid.  The page prints no values, so these pins use
exact hand-made fold cases (tests/golden), closed forms of SiLU, and values
from mpmath at 50 digits, an arbitrary-precision library independent of
numpy's exp.
"""
import json
import os

import mpmath
import numpy as np
import pytest

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
mpmath.mp.dps = 50


def mp_silu(z):
    z = mpmath.mpf(float(z))
    return float(z / (1 + mpmath.exp(-z)))


def test_fold_hand_cases():
    with open(os.path.join(GOLDEN, "bn_fold_hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    for cs in cases:
        scale, bias = oracle.bn_fold([cs["gamma"]], [cs["beta"]], [cs["mean"]], [cs["var"]],
                                     cs["eps"])
        assert scale[0] == cs["scale"] and bias[0] == cs["bias"], cs


def test_fold_identity_statistics():
    """gamma=1, beta=0, mean=0, var=1: bias is exactly 0, scale is 1/sqrt(1+eps)."""
    eps = np.float32(1e-3)
    scale, bias = oracle.bn_fold(np.ones(4, np.float32), np.zeros(4, np.float32),
                                 np.zeros(4, np.float32), np.ones(4, np.float32), eps)
    assert np.all(bias == 0.0)
    exact = float(1 / mpmath.sqrt(1 + mpmath.mpf(float(eps))))
    assert np.all(np.abs(scale - exact) <= 2 * np.spacing(exact))


def test_fold_is_bn_of_a_value():
    """t*scale + bias equals gamma*(t-mean)/sqrt(var+eps) + beta evaluated at 50 digits."""
    rng = np.random.default_rng(3)
    g = rng.uniform(0.5, 1.5, 8).astype(np.float32)
    b = rng.normal(0, 0.1, 8).astype(np.float32)
    m = rng.normal(0, 0.1, 8).astype(np.float32)
    v = rng.uniform(0.5, 2, 8).astype(np.float32)
    eps = np.float32(1e-3)
    scale, bias = oracle.bn_fold(g, b, m, v, eps)
    for t in (-3.0, 0.0, 0.7, 5.0):
        for k in range(8):
            ref = (mpmath.mpf(float(g[k])) * (t - mpmath.mpf(float(m[k])))
                   / mpmath.sqrt(mpmath.mpf(float(v[k])) + mpmath.mpf(float(eps)))
                   + mpmath.mpf(float(b[k])))
            assert abs(t * scale[k] + bias[k] - float(ref)) <= 1e-14 * (1 + abs(float(ref)))


def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(30.0) - 30.0) < 1e-11          # SiLU(x) -> x for large x
    assert abs(oracle.silu(-30.0)) < 1e-11                 # SiLU(x) -> 0 for very negative x
    assert oracle.silu(-30.0) < 0
    big_neg = oracle.silu(-800.0)                          # exp overflows: limit is -0
    assert big_neg == 0.0 and np.signbit(big_neg)
    assert abs(oracle.silu(1.0) - mp_silu(1.0)) < 1e-16


def test_silu_odd_part_identity():
    """SiLU(x) - SiLU(-x) = x: sigmoid(x) + sigmoid(-x) = 1."""
    x = np.linspace(-12, 12, 97)
    np.testing.assert_allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=1e-14, atol=1e-14)


def test_silu_minimum_lambert_w():
    """The minimum of SiLU sits at x* = -1 - W(1/e) and its value is -W(1/e)."""
    w = float(mpmath.lambertw(mpmath.e ** -1).real)
    x_star = -1.0 - w
    val = oracle.silu(x_star)
    assert abs(val - (-w)) < 1e-15
    for h in (1e-3, 1e-2, 0.1):
        assert oracle.silu(x_star - h) > val and oracle.silu(x_star + h) > val


def test_silu_against_mpmath():
    zs = np.concatenate([np.linspace(-40, 40, 161), [-1e-8, 1e-8, 1e-300, 88.0, -88.0]])
    got = oracle.silu(zs)
    for z, g in zip(zs, got):
        ref = mp_silu(z)
        assert abs(g - ref) <= 4 * np.spacing(abs(ref)) + 1e-300, (z, g, ref)


def test_bn_of_folded_statistics_is_batchnorm():
    """oracle.bn with the folded scale/bias, channels last, equals the textbook
    gamma*(t-mean)/sqrt(var+eps) + beta per channel (50 digits); at t = mean it is beta."""
    rng = np.random.default_rng(4)
    g = rng.uniform(0.5, 1.5, 6).astype(np.float32)
    b = rng.normal(0, 0.1, 6).astype(np.float32)
    m = rng.normal(0, 0.1, 6).astype(np.float32)
    v = rng.uniform(0.5, 2, 6).astype(np.float32)
    eps = np.float32(1e-3)
    scale, bias = oracle.bn_fold(g, b, m, v, eps)
    t = rng.normal(0, 2, (3, 4, 6))
    got = oracle.bn(t, scale, bias)
    assert got.shape == t.shape
    for idx in np.ndindex(3, 4, 6):
        k = idx[-1]
        ref = (mpmath.mpf(float(g[k])) * (mpmath.mpf(float(t[idx])) - mpmath.mpf(float(m[k])))
               / mpmath.sqrt(mpmath.mpf(float(v[k])) + mpmath.mpf(float(eps))) + mpmath.mpf(float(b[k])))
        assert abs(got[idx] - float(ref)) <= 1e-14 * (1 + abs(float(ref))), idx
    at_mean = oracle.bn(np.broadcast_to(m.astype(np.float64), (2, 6)), scale, bias)
    np.testing.assert_allclose(at_mean, np.broadcast_to(b.astype(np.float64), (2, 6)), atol=1e-15)


def test_bn_silu_per_channel_broadcast():
    """Channel k (last axis) uses scale[k] and bias[k]; identity BN gives SiLU(conv)."""
    conv = np.arange(2 * 3 * 5, dtype=np.float64).reshape(2, 3, 5) / 7.0 - 2.0
    np.testing.assert_array_equal(oracle.bn_silu(conv, np.ones(5), np.zeros(5)), oracle.silu(conv))
    scale = np.array([1.0, -2.0, 0.5, 3.0, 0.0])
    bias = np.array([0.0, 1.0, -1.0, 0.25, 2.0])
    got = oracle.bn_silu(conv, scale, bias)
    for k in range(5):
        np.testing.assert_array_equal(got[..., k], oracle.silu(conv[..., k] * scale[k] + bias[k]))


def test_whole_layer_on_hand_case():
    """Hand-summed conv (golden case C) -> BN fold (golden fold case 1) -> SiLU at 50 digits."""
    with open(os.path.join(GOLDEN, "conv_hand_cases.json")) as f:
        doc = json.load(f)
    case = next(c for c in doc["cases"] if c["name"] == "C_2x2_pad1")
    x = f32_to_bf16_bits(np.asarray(doc["x_2x2x2"], np.float32))
    w = f32_to_bf16_bits(np.asarray(case["w"], np.float32))
    # channel 0: scale 1, bias 0.5 ; channel 1: scale 1, bias -2 (exact fold cases)
    gamma, beta, mean, var = [2.0, 3.0], [1.0, 0.0], [0.5, 2.0], [3.0, 8.0]
    y = oracle.conv_bn_silu(x, w, gamma, beta, mean, var, 1.0, case["stride"], case["pad"])
    conv = np.asarray(case["expected"], np.float64)
    bias = [0.5, -2.0]
    for idx in np.ndindex(conv.shape):
        ref = mp_silu(conv[idx] + bias[idx[-1]])
        assert abs(y[idx] - ref) <= 4 * np.spacing(abs(ref)) + 1e-300, idx


def test_sampled_whole_layer_matches_full():
    rng = np.random.default_rng(5)
    xb = f32_to_bf16_bits(rng.standard_normal((2, 7, 6, 4)).astype(np.float32))
    wb = f32_to_bf16_bits(rng.standard_normal((3, 3, 3, 4)).astype(np.float32) * 0.3)
    g, b = np.float32([1.1, 0.9, 1.3]), np.float32([0.1, -0.2, 0.0])
    m, v = np.float32([0.05, -0.1, 0.2]), np.float32([1.0, 0.7, 1.9])
    full = oracle.conv_bn_silu(xb, wb, g, b, m, v, 1e-3, 2, 1)
    pix = np.array([0, 5, 11, full.shape[1] * full.shape[2] * 2 - 1])
    at = oracle.conv_bn_silu_at(xb, wb, g, b, m, v, 1e-3, pix, 2, 1)
    np.testing.assert_array_equal(at, full.reshape(-1, 3)[pix])
