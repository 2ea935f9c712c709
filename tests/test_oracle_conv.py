"""Pins for the oracle's convolution (CPU only).

The fusion page ("Fusing an Epilogue", section "The problem") names the
convolution but prints no formula or values, so the oracle's conv is pinned
to things fixed outside it: hand sums on paper (tests/golden), closed forms,
an independent library routine (torch's float64 CPU conv2d, numpy matmul),
and identities of the mathematics (delta kernel, subsampling, linearity,
channel permutation).  Each pin is chosen to catch a specific plausible bug:
a swapped r/s or h/w index, a wrong sign of the padding offset, a dropped
tap, a stride applied to the wrong axis, a transposed weight operand.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "conv_hand_cases.json")


def bits(a):
    """Small integers or bf16-representable values -> bf16 bit patterns (exact)."""
    a = np.asarray(a, dtype=np.float32)
    b = f32_to_bf16_bits(a)
    assert np.array_equal(bf16_bits_to_f32(b), a), "fixture value not exact in bf16"
    return b


def load_cases():
    with open(GOLDEN) as f:
        doc = json.load(f)
    for case in doc["cases"]:
        x = doc[case["x"]] if isinstance(case["x"], str) else case["x"]
        yield pytest.param(x, case, id=case["name"])


@pytest.mark.parametrize("x,case", list(load_cases()))
def test_hand_summed_fixtures(x, case):
    out = oracle.conv2d(bits(x), bits(case["w"]), case["stride"], case["pad"], threads=1)
    expected = np.asarray(case["expected"], dtype=np.float64)
    assert out.shape == expected.shape
    assert np.array_equal(out, expected)


def test_all_ones_closed_form():
    """All-ones x and W, 3x3, pad 1, stride 1: a corner sees 4 taps, an edge 6, the inside 9."""
    c, h, w = 5, 6, 7
    x = bits(np.ones((1, h, w, c)))
    wt = bits(np.ones((2, 3, 3, c)))
    out = oracle.conv2d(x, wt, 1, 1)
    taps = np.full((h, w), 9.0)
    taps[0, :] = taps[-1, :] = 6
    taps[:, 0] = taps[:, -1] = 6
    taps[0, 0] = taps[0, -1] = taps[-1, 0] = taps[-1, -1] = 4
    for k in range(2):
        assert np.array_equal(out[0, :, :, k], taps * c)
    # stride 2 visits every other output of the stride-1 result
    out2 = oracle.conv2d(x, wt, 2, 1)
    assert np.array_equal(out2[0, :, :, 0], taps[::2, ::2] * c)


def rand_bits(rng, shape, scale=1.0):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * scale)


def torch_conv_f64(x_bits, w_bits, stride, pad):
    x = torch.from_numpy(bf16_bits_to_f32(x_bits).astype(np.float64)).permute(0, 3, 1, 2)
    w = torch.from_numpy(bf16_bits_to_f32(w_bits).astype(np.float64)).permute(0, 3, 1, 2)
    y = torch.nn.functional.conv2d(x, w, stride=stride, padding=pad)
    return y.permute(0, 2, 3, 1).contiguous().numpy()


@pytest.mark.parametrize("n,h,w,c,k,r,s,stride,pad", [
    (1, 8, 8, 3, 4, 3, 3, (1, 1), (1, 1)),
    (2, 9, 7, 5, 6, 3, 3, (2, 2), (1, 1)),
    (1, 11, 10, 4, 3, 5, 5, (2, 2), (2, 2)),
    (3, 6, 9, 2, 5, 2, 3, (1, 2), (0, 1)),
    (1, 7, 5, 8, 2, 1, 1, (1, 1), (0, 0)),
    (2, 5, 6, 3, 7, 3, 1, (2, 1), (1, 0)),
    (1, 3, 3, 4, 4, 3, 3, (3, 3), (2, 2)),
])
def test_matches_torch_float64_conv2d(n, h, w, c, k, r, s, stride, pad):
    """An independent library convolution (torch CPU, float64) on the same values."""
    rng = np.random.default_rng(1234 + n * 100 + h * 10 + w)
    xb = rand_bits(rng, (n, h, w, c))
    wb = rand_bits(rng, (k, r, s, c))
    out = oracle.conv2d(xb, wb, stride, pad)
    ref = torch_conv_f64(xb, wb, stride, pad)
    assert out.shape == ref.shape
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_pointwise_is_matmul():
    """A 1x1, stride-1 convolution is the plain product X[M, C] @ W[K, C]^T."""
    rng = np.random.default_rng(7)
    xb = rand_bits(rng, (2, 5, 4, 12))
    wb = rand_bits(rng, (9, 1, 1, 12))
    out = oracle.conv2d(xb, wb, 1, 0)
    xm = bf16_bits_to_f32(xb).astype(np.float64).reshape(-1, 12)
    wm = bf16_bits_to_f32(wb).astype(np.float64).reshape(9, 12)
    np.testing.assert_allclose(out.reshape(-1, 9), xm @ wm.T, rtol=1e-13, atol=1e-13)


def test_delta_kernel_is_identity():
    """A 3x3 kernel that is 1 only at its centre for k == c copies x through (pad 1)."""
    rng = np.random.default_rng(8)
    c = 6
    xb = rand_bits(rng, (2, 7, 5, c))
    wt = np.zeros((c, 3, 3, c), np.float32)
    for k in range(c):
        wt[k, 1, 1, k] = 1.0
    out = oracle.conv2d(xb, bits(wt), 1, 1)
    assert np.array_equal(out, bf16_bits_to_f32(xb).astype(np.float64))


def test_shifted_delta_moves_the_image():
    """A delta at tap (r, s) = (0, 2) reads x[h-1, w+1]: catches a swapped or negated offset."""
    rng = np.random.default_rng(9)
    xb = rand_bits(rng, (1, 6, 8, 1))
    wt = np.zeros((1, 3, 3, 1), np.float32)
    wt[0, 0, 2, 0] = 1.0
    out = oracle.conv2d(xb, bits(wt), 1, 1)[0, :, :, 0]
    xv = bf16_bits_to_f32(xb)[0, :, :, 0].astype(np.float64)
    exp = np.zeros_like(xv)
    exp[1:, :-1] = xv[:-1, 1:]
    assert np.array_equal(out, exp)


def test_stride2_is_subsampled_stride1():
    rng = np.random.default_rng(10)
    xb = rand_bits(rng, (2, 9, 10, 3))
    wb = rand_bits(rng, (4, 3, 3, 3))
    full = oracle.conv2d(xb, wb, 1, 1)
    strided = oracle.conv2d(xb, wb, 2, 1)
    assert np.array_equal(strided, full[:, ::2, ::2, :])


def test_linearity_exact():
    """conv(2*x1 - x2, W) = 2*conv(x1, W) - conv(x2, W), exactly on small integers."""
    rng = np.random.default_rng(11)
    x1 = rng.integers(-4, 5, (1, 6, 6, 3)).astype(np.float32)
    x2 = rng.integers(-4, 5, (1, 6, 6, 3)).astype(np.float32)
    w1 = rng.integers(-3, 4, (5, 3, 3, 3)).astype(np.float32)
    w2 = rng.integers(-3, 4, (5, 3, 3, 3)).astype(np.float32)
    c = lambda x, w: oracle.conv2d(bits(x), bits(w), 1, 1)
    assert np.array_equal(c(2 * x1 - x2, w1), 2 * c(x1, w1) - c(x2, w1))
    assert np.array_equal(c(x1, 3 * w1 + w2), 3 * c(x1, w1) + c(x1, w2))


def test_output_channel_permutation():
    rng = np.random.default_rng(12)
    xb = rand_bits(rng, (1, 5, 5, 4))
    wb = rand_bits(rng, (6, 3, 3, 4))
    perm = rng.permutation(6)
    a = oracle.conv2d(xb, wb, 1, 1)
    b = oracle.conv2d(xb, wb[perm], 1, 1)
    assert np.array_equal(b, a[..., perm])


def test_sampled_pixels_match_full_and_threads_do_not_change_results():
    rng = np.random.default_rng(13)
    xb = rand_bits(rng, (3, 9, 8, 5))
    wb = rand_bits(rng, (7, 3, 3, 5))
    full1 = oracle.conv2d(xb, wb, 2, 1, threads=1)
    fullt = oracle.conv2d(xb, wb, 2, 1, threads=5)
    assert np.array_equal(full1, fullt)
    flat = full1.reshape(-1, 7)
    pix = rng.choice(flat.shape[0], 20, replace=False)
    at = oracle.conv2d_at(xb, wb, pix, 2, 1, threads=3)
    assert np.array_equal(at, flat[pix])


def test_invalid_shapes_rejected():
    xb = np.zeros((1, 2, 2, 1), np.uint16)
    wb = np.zeros((1, 3, 3, 1), np.uint16)
    with pytest.raises(ValueError):
        oracle.conv2d(xb, wb, 1, 0)     # kernel larger than the padded image
    with pytest.raises(ValueError):
        oracle.conv2d_at(xb, wb, np.array([4]), 1, 1)  # pixel index out of range
