"""The thin-input tensor-core kernel (3x3 filters over 1, 3 or 4 channels) against the
oracle, every element (GPU only).

The kernel gives each CTA an equal contiguous range of output pixels and stages
the input rows that range reads in shared memory with bulk copies (plain loads
for an unaligned head or tail), in passes of whole output rows when they do not
all fit at once.  These shapes reach each of those cases: rows whose byte length
is not a multiple of 16 (and rows shorter than 16 bytes), ranges that cross
images, wide rows that force one output row per pass and several passes per CTA,
a batch of stems, strides 1-3, paddings 0-2, and output channel counts below,
at and between the kernel's N widths.
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


CASES = [
    # n, h, w, c, c_out, stride, pad
    (3, 11, 13, 3, 24, 1, 1),       # 78-byte rows: unaligned head and tail
    (2, 9, 7, 1, 8, 2, 0),          # 14-byte rows: runs shorter than 16 bytes
    (5, 6, 6, 4, 64, 1, 2),         # pad 2, ranges across images, N = 64
    (2, 50, 50, 3, 16, 3, 0),       # stride 3
    (1, 30, 30, 1, 48, 2, 1),       # N = 48
    (2, 33, 17, 4, 40, 1, 0),       # c = 4 (K 36 -> 64), c_out between N widths
    (1, 12, 1800, 3, 16, 1, 1),     # 10.8 KB rows, the widest that fit: one output row per staging pass
    (4, 64, 1500, 3, 16, 1, 1),     # 9 KB rows: several passes per CTA
    (8, 640, 640, 3, 16, 2, 1),     # a batch of YOLO stems: shares of 2695 pixels, passes of 4 rows
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}-s{c[5]}p{c[6]}"
                                             for c in CASES])
def test_thin_input_kernel_matches_oracle(capi, case):
    n, h, w, c, k, stride, pad = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = capi.plan(n, h, w, c, k, 3, 3, stride, pad, "auto", sms)
    assert p["algo"] == "tcgen05" and p["threads"] == 288, p    # the thin-input kernel
    inp = make_layer_inputs(LayerShape("thin", n, h, w, c, k, 3, 3, stride, pad), seed=500 + n * c)
    dev = torch.device("cuda:0")
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    wt = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    y = capi.forward(x, wt, scale, bias, stride, pad)
    torch.cuda.synchronize()
    capi.check()
    got = bf16_bits_to_f32(torch_bf16_to_bits(y)).astype(np.float64)
    ref = oracle.conv_bn_silu(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var, inp.eps,
                              stride, pad)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{case}: {int(bad.sum())} of {bad.size} out of tolerance; worst at {idx}: "
                             f"gpu {got[idx]!r} oracle {ref[idx]!r}")
    # A second run is bit-identical (no atomics; fixed per-pixel arithmetic).
    y2 = capi.forward(x, wt, scale, bias, stride, pad)
    torch.cuda.synchronize()
    assert np.array_equal(torch_bf16_to_bits(y), torch_bf16_to_bits(y2))
