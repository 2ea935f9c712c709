"""Pins for the oracle's other epilogues (CPU only): identity and ReLU after the
BN multiply/add, and a residual added after the activation.

"Fusing an Epilogue", section "What an epilogue is", names activations and bias
adds as element-wise epilogue work; it prints no values.  The pins are a
hand-derived fixture on a hand-summed convolution (tests/golden), closed forms
of ReLU, and consistency with the SiLU layer and with the sampled-pixel path.
"""
import json
import os

import numpy as np
import pytest

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(a):
    a = np.asarray(a, dtype=np.float32)
    b = f32_to_bf16_bits(a)
    assert np.array_equal(bf16_bits_to_f32(b), a), "fixture value not exact in bf16"
    return b


def load():
    with open(os.path.join(GOLDEN, "epilogue_hand_cases.json")) as f:
        ep = json.load(f)
    with open(os.path.join(GOLDEN, "conv_hand_cases.json")) as f:
        conv = json.load(f)
    case = next(c for c in conv["cases"] if c["name"] == ep["conv_case"])
    x = conv[case["x"]] if isinstance(case["x"], str) else case["x"]
    return ep, case, x


EP, CONV_CASE, CONV_X = load()


@pytest.mark.parametrize("case", EP["cases"], ids=[c["name"] for c in EP["cases"]])
def test_hand_derived_epilogues(case):
    expected = np.asarray(case["expected"], dtype=np.float64)
    res = None
    if case["residual"]:
        res = bits(np.broadcast_to(np.asarray(EP["residual_per_channel"], np.float32), expected.shape))
    got = oracle.conv_bn_act(bits(CONV_X), bits(CONV_CASE["w"]), np.float32(EP["gamma"]),
                             np.float32(EP["beta"]), np.float32(EP["mean"]), np.float32(EP["var"]),
                             EP["eps"], CONV_CASE["stride"], CONV_CASE["pad"], case["activation"], res, threads=1)
    assert got.shape == expected.shape
    assert np.array_equal(got, expected), case["name"]


def test_relu_closed_forms():
    z = np.array([-3.5, -1e-300, -0.0, 0.0, 1e-300, 2.25, 1e300])
    r = oracle.relu(z)
    assert np.array_equal(r, (z + np.abs(z)) / 2)              # (z + |z|)/2
    assert np.array_equal(r - oracle.relu(-z), z)               # relu(z) - relu(-z) = z
    assert np.all(r >= 0)


def test_silu_without_residual_is_the_layer():
    rng = np.random.default_rng(5)
    xb = f32_to_bf16_bits(rng.standard_normal((2, 6, 5, 8)).astype(np.float32))
    wb = f32_to_bf16_bits(rng.standard_normal((4, 3, 3, 8)).astype(np.float32) * 0.2)
    g, b = rng.uniform(0.5, 1.5, 4), rng.normal(0, 0.1, 4)
    m, v = rng.normal(0, 0.1, 4), rng.uniform(0.5, 2, 4)
    a = oracle.conv_bn_act(xb, wb, g, b, m, v, 1e-3, 1, 1, "silu")
    assert np.array_equal(a, oracle.conv_bn_silu(xb, wb, g, b, m, v, 1e-3, 1, 1))
    ident = oracle.conv_bn_act(xb, wb, g, b, m, v, 1e-3, 1, 1, "identity")
    sc, bi = oracle.bn_fold(g, b, m, v, 1e-3)
    assert np.array_equal(ident, oracle.bn(oracle.conv2d(xb, wb, 1, 1), sc, bi))
    assert np.array_equal(a, oracle.silu(ident))


def test_sampled_pixels_take_their_residual_rows():
    rng = np.random.default_rng(6)
    xb = f32_to_bf16_bits(rng.standard_normal((2, 7, 6, 8)).astype(np.float32))
    wb = f32_to_bf16_bits(rng.standard_normal((5, 3, 3, 8)).astype(np.float32) * 0.2)
    rb = f32_to_bf16_bits(rng.standard_normal((2, 4, 3, 5)).astype(np.float32))
    g, b = np.ones(5), np.zeros(5)
    m, v = np.zeros(5), np.ones(5)
    full = oracle.conv_bn_act(xb, wb, g, b, m, v, 0.0, 2, 1, "relu", rb).reshape(-1, 5)
    pix = np.array([0, 5, 7, 23, 11])
    at = oracle.conv_bn_act_at(xb, wb, g, b, m, v, 0.0, pix, 2, 1, "relu", rb)
    assert np.array_equal(at, full[pix])


def test_unknown_activation_rejected():
    with pytest.raises(ValueError):
        oracle.activate(np.zeros(2), "gelu")
