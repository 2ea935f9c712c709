"""Parity of the CUDA path with the fp64 CPU oracle, through the C ABI (GPU only).

Every case draws seeded synthetic inputs, runs the BN fold and the fused
forward on the GPU, and compares every output element with the oracle:
|y_gpu - y_oracle| <= 1e-2 + 1e-2 * |y_oracle| (the bf16-output tolerance the
layer is specified with).  The oracle folds BN in float64 from the same
gamma/beta/mean/var; nothing it uses comes from the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import (LAYERS, LAYER_ORDER, LayerShape,
                                                   bf16_bits_to_f32, bits_to_torch_bf16,
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


def to_dev(inp):
    dev = torch.device("cuda:0")
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    stats = [torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var)]
    return x, w, stats


def run_gpu(capi, inp, algo="auto", stride=None, pad=None):
    sh = inp.shape
    x, w, (g, b, m, v) = to_dev(inp)
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    y = capi.forward(x, w, scale, bias, sh.stride if stride is None else stride,
                     sh.pad if pad is None else pad, algo=algo)
    torch.cuda.synchronize()
    capi.check()
    return y


def y_to_f64(y):
    return bf16_bits_to_f32(torch_bf16_to_bits(y)).astype(np.float64)


def assert_parity(got, ref, what):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"worst at {idx}: gpu {got[idx]!r} oracle {ref[idx]!r}")


def oracle_full(inp, stride=None, pad=None):
    sh = inp.shape
    return oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var,
                               inp.eps, sh.stride if stride is None else stride,
                               sh.pad if pad is None else pad)


# ------------------------------------------------------------------ BN fold
def test_fold_matches_oracle(capi):
    for name in LAYER_ORDER:
        inp = make_layer_inputs(LAYERS[name])
        _, _, (g, b, m, v) = to_dev(inp)
        scale, bias = capi.fold(g, b, m, v, inp.eps)
        torch.cuda.synchronize()
        ref_s, ref_b = oracle.bn_fold(inp.gamma, inp.beta, inp.mean, inp.var, inp.eps)
        gs = scale.cpu().numpy().astype(np.float64)
        gb = bias.cpu().numpy().astype(np.float64)
        # one rounding to fp32 of a float64 result: within one fp32 ulp of the exact value
        assert np.all(np.abs(gs - ref_s) <= np.spacing(np.abs(ref_s).astype(np.float32))), name
        assert np.all(np.abs(gb - ref_b) <= 2 * np.spacing(np.abs(ref_b).astype(np.float32))), name


def test_fold_batch_is_bit_identical_to_single_folds(capi):
    """One batched launch over the five layers (plus an empty one) gives exactly the
    scale/bias of the per-layer fold."""
    layers, singles = [], []
    for name in LAYER_ORDER:
        inp = make_layer_inputs(LAYERS[name])
        _, _, (g, b, m, v) = to_dev(inp)
        s1, b1 = capi.fold(g, b, m, v, inp.eps)
        singles.append((s1, b1))
        layers.append((g, b, m, v, inp.eps, torch.full_like(s1, float("nan")), torch.full_like(b1, float("nan"))))
    empty = torch.empty(0, dtype=torch.float32, device="cuda:0")
    capi.fold_batch(layers[:2] + [(empty, empty, empty, empty, 1e-3, empty, empty)] + layers[2:])
    torch.cuda.synchronize()
    for (s1, b1), lay in zip(singles, layers):
        assert torch.equal(s1, lay[5]) and torch.equal(b1, lay[6])


# ------------------------------------------------------------------ the five layers, full size
@pytest.mark.parametrize("name", LAYER_ORDER)
def test_layer_full_size_default_kernel(capi, name):
    inp = make_layer_inputs(LAYERS[name])
    y = run_gpu(capi, inp)
    assert_parity(y_to_f64(y), oracle_full(inp), f"{name} (auto)")


@pytest.mark.parametrize("name", ["tiny", "down", "pointwise", "deep"])
def test_layer_full_size_tcgen05_kernel(capi, name):
    inp = make_layer_inputs(LAYERS[name])
    y = run_gpu(capi, inp, algo="tcgen05")
    assert_parity(y_to_f64(y), oracle_full(inp), f"{name} (tcgen05)")


@pytest.mark.parametrize("name", ["tiny", "stem", "pointwise"])
def test_layer_full_size_direct_kernel(capi, name):
    inp = make_layer_inputs(LAYERS[name])
    y = run_gpu(capi, inp, algo="direct")
    assert_parity(y_to_f64(y), oracle_full(inp), f"{name} (direct)")


@pytest.mark.parametrize("name", ["down", "deep"])
def test_layer_full_size_direct_kernel_sampled(capi, name):
    inp = make_layer_inputs(LAYERS[name])
    sh = inp.shape
    y = y_to_f64(run_gpu(capi, inp, algo="direct")).reshape(-1, sh.k)
    rng = np.random.default_rng(17)
    pix = np.unique(np.concatenate([rng.choice(sh.m, 3000, replace=False), [0, sh.m - 1]]))
    ref = oracle.conv_bn_silu_at(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var,
                                 inp.eps, pix, sh.stride, sh.pad)
    assert_parity(y[pix], ref, f"{name} (direct, sampled)")


@pytest.mark.parametrize("name", LAYER_ORDER)
def test_deterministic(capi, name):
    inp = make_layer_inputs(LAYERS[name])
    a = torch_bf16_to_bits(run_gpu(capi, inp))
    b = torch_bf16_to_bits(run_gpu(capi, inp))
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ shape sweep
SWEEP = [
    # n, h, w, c, k, r, s, stride, pad
    (1, 7, 9, 16, 32, 3, 3, 1, 1),      # odd image, M=63 < one tile
    (2, 13, 11, 16, 24, 3, 3, 1, 1),    # c_out not a multiple of the tile
    (3, 17, 19, 32, 48, 3, 3, 2, 1),    # stride 2, odd sizes, tiles cross images
    (2, 15, 15, 64, 64, 3, 3, 2, 1),
    (1, 11, 10, 48, 40, 3, 3, 1, 1),    # c = 48 -> 16-channel K steps
    (2, 9, 9, 96, 72, 3, 3, 1, 1),      # c = 96 -> 32-channel K steps
    (4, 8, 8, 128, 136, 3, 3, 1, 1),    # c_out just above a 128 tile
    (1, 12, 12, 64, 264, 1, 1, 1, 0),   # c_out > 256: several N tiles with a tail
    (2, 14, 14, 64, 32, 5, 5, 1, 2),    # 5x5 filter
    (2, 10, 10, 32, 16, 5, 5, 2, 2),
    (1, 1, 1, 16, 16, 3, 3, 1, 1),      # a single pixel: all but the centre tap padded
    (3, 5, 5, 16, 8, 1, 1, 1, 0),       # c_out = 8 < smallest tile
    (1, 6, 6, 16, 16, 3, 3, 3, 0),      # stride larger than needed
    (1, 9, 9, 16, 16, 3, 3, 2, 0),      # no padding, stride 2
    (2, 8, 8, 3, 16, 3, 3, 2, 1),       # 3-channel stem shape (thin-input tensor-core kernel)
    (2, 13, 11, 4, 24, 3, 3, 1, 1),     # c = 4 (K 36 -> 64), c_out 24 in a 32-wide tile
    (1, 30, 30, 1, 48, 3, 3, 2, 1),     # c = 1, N = 48
    (1, 33, 17, 3, 64, 3, 3, 1, 0),     # c = 3, N = 64, no padding
    (1, 9, 7, 8, 8, 3, 3, 1, 1),        # c = 8 (direct)
    (2, 9, 7, 24, 20, 3, 3, 1, 1),      # c = 24, c_out = 20 (direct)
    (2, 9, 8, 16, 16, 3, 1, (1, 2), (1, 0)),  # asymmetric filter/stride/pad
    (1, 64, 64, 16, 16, 3, 3, 1, 1),    # 32 tiles of 128 pixels
    (64, 20, 20, 64, 64, 3, 3, 1, 1),   # 200 M tiles: several tiles per CTA, TMEM double buffer
]


@pytest.mark.parametrize("case", SWEEP, ids=[str(i) for i in range(len(SWEEP))])
@pytest.mark.parametrize("algo", ["auto", "direct", "tcgen05"])
def test_shape_sweep(capi, case, algo):
    n, h, w, c, k, r, s, stride, pad = case
    if algo == "tcgen05":
        try:
            capi.plan(n, h, w, c, k, r, s, stride, pad, "tcgen05")
        except capi.CbsError:
            pytest.skip("shape outside the tensor-core kernel")
    shape = LayerShape("sweep", n, h, w, c, k, r, s, 1, 0)
    inp = make_layer_inputs(shape, seed=1000 + hash(case) % 1000)
    y = run_gpu(capi, inp, algo=algo, stride=stride, pad=pad)
    assert_parity(y_to_f64(y), oracle_full(inp, stride, pad), f"{case} ({algo})")


def test_forced_tcgen05_on_supported_shapes(capi):
    """The tensor-core kernel itself (not the automatic choice) on a few shapes."""
    for case in [(2, 13, 11, 16, 24, 3, 3, 1, 1), (1, 12, 12, 64, 264, 1, 1, 1, 0),
                 (3, 17, 19, 32, 48, 3, 3, 2, 1)]:
        n, h, w, c, k, r, s, stride, pad = case
        inp = make_layer_inputs(LayerShape("forced", n, h, w, c, k, r, s, stride, pad), seed=77)
        y = run_gpu(capi, inp, algo="tcgen05")
        assert_parity(y_to_f64(y), oracle_full(inp), f"{case} (tcgen05)")


# ------------------------------------------------------------------ edge cases
def test_empty_batch_is_a_noop(capi):
    dev = torch.device("cuda:0")
    x = torch.empty((0, 8, 8, 16), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((16, 3, 3, 16), dtype=torch.bfloat16, device=dev)
    s = torch.ones(16, device=dev)
    y = capi.forward(x, w, s, s, 1, 1)
    assert y.shape == (0, 8, 8, 16)


def test_large_values_saturate_like_silu(capi):
    """Huge positive outputs pass through, huge negative ones go to (minus) zero."""
    shape = LayerShape("sat", 1, 8, 8, 16, 16, 1, 1, 1, 0)
    inp = make_layer_inputs(shape, seed=5)
    inp.gamma[:] = 1.0
    inp.var[:] = 1.0
    inp.mean[:] = 0.0
    inp.beta[:8] = 200.0
    inp.beta[8:] = -200.0
    y = y_to_f64(run_gpu(capi, inp))
    ref = oracle_full(inp)
    assert_parity(y, ref, "saturation")
    assert np.all(y[..., 8:] <= 0) and np.all(np.abs(y[..., 8:]) < 1e-6)


def test_misaligned_pointer_rejected(capi):
    dev = torch.device("cuda:0")
    buf = torch.zeros(4096, dtype=torch.bfloat16, device=dev)
    w = torch.zeros((16, 1, 1, 16), dtype=torch.bfloat16, device=dev)
    s = torch.ones(16, device=dev)
    y = torch.empty((1, 4, 4, 16), dtype=torch.bfloat16, device=dev)
    with pytest.raises(capi.CbsError) as e:
        capi.forward_ptr(buf.data_ptr() + 2, w.data_ptr(), s.data_ptr(), s.data_ptr(), y.data_ptr(),
                         1, 4, 4, 16, 16, 1, 1, 1, 0)
    assert e.value.status == capi.CBS_ERR_MISALIGNED


def test_streams_are_honoured(capi):
    """A call on a side stream is ordered on that stream."""
    inp = make_layer_inputs(LAYERS["tiny"])
    x, w, (g, b, m, v) = to_dev(inp)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        scale, bias = capi.fold(g, b, m, v, inp.eps)
        y = capi.forward(x, w, scale, bias, 1, 1)
    side.synchronize()
    capi.check(side)
    assert_parity(y_to_f64(y), oracle_full(inp), "side stream")


def test_silu_over_a_wide_range(capi):
    """A 1x1 conv that copies one channel makes z sweep [-120, 120]: the epilogue's SiLU
    must match the oracle over the whole range (saturation on both sides included)."""
    from conv2d_batchnorm_silu_gb300.synthetic import f32_to_bf16_bits
    shape = LayerShape("silu", 1, 64, 64, 16, 16, 1, 1, 1, 0)
    inp = make_layer_inputs(shape, seed=9)
    x = np.zeros((1, 64, 64, 16), np.float32)
    x[..., 0] = np.linspace(-120.0, 120.0, 64 * 64, dtype=np.float32).reshape(64, 64)
    x[..., 1] = np.linspace(-6.0, 6.0, 64 * 64, dtype=np.float32).reshape(64, 64)
    w = np.zeros((16, 1, 1, 16), np.float32)
    w[:8, 0, 0, 0] = 1.0
    w[8:, 0, 0, 1] = 1.0
    inp.x_bits = f32_to_bf16_bits(x)
    inp.w_bits = f32_to_bf16_bits(w)
    inp.gamma[:] = 1.0
    inp.beta[:] = 0.0
    inp.mean[:] = 0.0
    inp.var[:] = 1.0
    inp.eps = 0.0
    for algo in ("auto", "direct"):
        y = y_to_f64(run_gpu(capi, inp, algo=algo))
        assert_parity(y, oracle_full(inp), f"SiLU sweep ({algo})")


STREAM_K_CASES = [
    # n, h, w, c, k, r, s, stride, pad: more 128x256 tiles than SMs, K loop >= 16 steps
    (32, 20, 20, 128, 512, 3, 3, 1, 1),   # 200 tiles, 18 K steps
    (39, 20, 20, 256, 384, 3, 3, 1, 1),   # 244 tiles, ragged last M tile, a 128-channel N tail
    (31, 20, 20, 128, 512, 3, 3, 1, 1),   # 97 M tiles: the last CTA pair's odd half is past the end
    # 2-CTA pairs whose second 256-channel tile is mostly past c_out: chunks with no channel are
    # neither published nor combined (per-chunk stream-K flags), on units split three ways and,
    # for each worker's last unit, four ways
    (33, 20, 20, 128, 264, 3, 3, 1, 1),   # an 8-channel N tail and a ragged M tail
    (32, 20, 20, 128, 320, 3, 3, 1, 1),   # a 64-channel N tail
]


@pytest.mark.parametrize("case", STREAM_K_CASES,
                         ids=["200tiles", "244tiles_ragged", "odd_m_tiles", "n_tail_8", "n_tail_64"])
def test_stream_k_split_tiles(capi, case):
    """Shapes whose plan splits the K loop of some tiles between two CTAs (stream-K):
    every output matches the oracle and two runs are bit-identical (the partial sums
    are combined in a fixed order and the ready flags return to zero)."""
    n, h, w, c, k, r, s, stride, pad = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = capi.plan(n, h, w, c, k, r, s, stride, pad, "auto", sms)
    assert p["algo"] == "tcgen05" and p["stream_k"] == 1 and p["block_n"] == 256, p
    inp = make_layer_inputs(LayerShape("streamk", n, h, w, c, k, r, s, stride, pad), seed=31)
    y1 = run_gpu(capi, inp)
    y2 = run_gpu(capi, inp)
    assert np.array_equal(torch_bf16_to_bits(y1), torch_bf16_to_bits(y2))
    assert_parity(y_to_f64(y1), oracle_full(inp), f"{case} (stream-K)")


SWAP_AB_CASES = [
    # n, h, w, c, k, r, s, stride, pad: 65..256 output channels, many 256-pixel tiles
    (1, 210, 190, 16, 80, 3, 3, 1, 1),    # channel tail (80 of 128), ragged last pixel tile
    (2, 280, 280, 64, 128, 3, 3, 2, 1),   # stride 2, 32-pixel last tile
    (1, 150, 150, 32, 200, 3, 3, 1, 1),   # two channel tiles, the second 72 wide
]


@pytest.mark.parametrize("case", SWAP_AB_CASES, ids=["c80_ragged", "s2_c128", "c200_two_tiles"])
def test_swap_ab_tiles(capi, case):
    """Shapes planned as channels x pixels tiles (MMA at N = 256, transposing epilogue)."""
    n, h, w, c, k, r, s, stride, pad = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = capi.plan(n, h, w, c, k, r, s, stride, pad, "auto", sms)
    assert p["algo"] == "tcgen05" and p["swap_ab"] == 1, p
    inp = make_layer_inputs(LayerShape("swap", n, h, w, c, k, r, s, stride, pad), seed=41)
    y1 = run_gpu(capi, inp)
    y2 = run_gpu(capi, inp)
    assert np.array_equal(torch_bf16_to_bits(y1), torch_bf16_to_bits(y2))
    assert_parity(y_to_f64(y1), oracle_full(inp), f"{case} (swap AB)")
