"""fp8 e4m3 output on the GPU (conv_bn_act_forward_fp8): the narrower output
cast of "Fusing an Epilogue", section "What an epilogue is".  Every element
is compared with the oracle's value: the GPU's one rounding from its fp32
result to e4m3 may land one code away from the oracle's rounding of the exact
value only when the two sit on either side of a rounding boundary, so the bound
is half an e4m3 step (2^-4 relative, 2^-10 absolute below 2^-6) plus the fp32
path's own error; and at least 99 % of the codes must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import LayerShape, bits_to_torch_bf16, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from conv2d_batchnorm_silu_gb300 import _build
    _build.build()
    from conv2d_batchnorm_silu_gb300 import capi as c
    return c


SHAPES = [
    LayerShape("tiny", 1, 32, 32, 16, 32, 3, 3, 1, 1),           # 32-byte fp8 rows (swizzled)
    LayerShape("n16", 2, 17, 19, 16, 16, 3, 3, 2, 1),            # 16-byte fp8 rows
    LayerShape("down", 2, 80, 80, 64, 128, 3, 3, 2, 1),          # pixel-major, 128-wide tiles
    LayerShape("c2f", 8, 80, 80, 128, 128, 1, 1, 1, 0),          # channel-major (swap AB), balanced 32-pixel runs
    LayerShape("swapw", 16, 160, 160, 16, 64, 3, 3, 2, 1),       # channel-major, whole 256-pixel tiles
    LayerShape("pairs", 31, 20, 20, 128, 512, 3, 3, 1, 1),       # 2-CTA stream-K
    LayerShape("stem", 1, 64, 64, 3, 16, 3, 3, 2, 1),            # direct kernel
    LayerShape("odd", 1, 9, 7, 16, 24, 3, 3, 1, 1),              # c_out % 16 != 0: direct kernel
]
CASES = [(s, a) for s in SHAPES for a in ("silu", "relu", "identity")]


@pytest.mark.parametrize("shape,activation", CASES, ids=[f"{s.name}-{a}" for s, a in CASES])
def test_fp8_output_matches_oracle(capi, shape, activation):
    dev = torch.device("cuda:0")
    inp = make_layer_inputs(shape, seed=29)
    x = bits_to_torch_bf16(inp.x_bits).to(dev)
    w = bits_to_torch_bf16(inp.w_bits).to(dev)
    g, b, m, v = (torch.from_numpy(a).to(dev) for a in (inp.gamma, inp.beta, inp.mean, inp.var))
    scale, bias = capi.fold(g, b, m, v, inp.eps)
    # a wide output range, so that the largest values saturate at 448: scale the BN by 200
    scale = scale * 200.0
    bias = bias * 200.0
    y = capi.forward_act_fp8(x, w, scale, bias, shape.stride, shape.pad, activation=activation)
    torch.cuda.synchronize()
    capi.check()
    got_codes = y.cpu().numpy()
    got = oracle.e4m3_bits_to_f64(got_codes)
    conv = oracle.conv2d(inp.x_bits, inp.w_bits, shape.stride, shape.pad)
    ref = oracle.bn_act(conv, scale.cpu().numpy().astype(np.float64), bias.cpu().numpy().astype(np.float64),
                        activation)
    clipped = np.clip(ref, -oracle.E4M3_MAX, oracle.E4M3_MAX)
    bound = 2.0 ** -4 * np.abs(clipped) + 2.0 ** -10 + 1e-3 * (1 + np.abs(clipped))
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - clipped) <= bound), float((np.abs(got - clipped) - bound).max())
    exact = oracle.to_e4m3_bits(ref)
    same = np.mean((got_codes == exact) | (got == oracle.e4m3_bits_to_f64(exact)))
    assert same >= 0.99, same
    if activation == "identity":
        assert np.any(np.abs(ref) > oracle.E4M3_MAX), "the case should exercise saturation"
