"""Seeded synthetic inputs for the fused conv2d -> BN -> SiLU layer.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds none of the layer's arithmetic: it only draws
random numbers and rounds them to the storage types (bf16 for activations
and weights, fp32 for the BatchNorm statistics).

Recipe (the same for every layer shape):

* x ~ N(0, 1), drawn in fp32 then rounded to bf16 (round to nearest even);
* W ~ N(0, var = 2 / fan_in) with fan_in = C*R*S (Kaiming normal), drawn in
  fp32 then rounded to bf16;
* gamma ~ U(0.5, 1.5), beta ~ N(0, 0.1), running mean ~ N(0, 0.1),
  running var ~ U(0.5, 2) (the 0.1 is a standard deviation), all fp32;
* eps = 1e-3.

The generator is numpy's PCG64, seeded per layer; x, W and each BN vector
come from their own child stream of one ``SeedSequence`` so that changing one
shape does not shift the others.  Arrays come back in NHWC / KRSC layout;
bf16 tensors are returned as their uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class LayerShape:
    """One convolution layer: NHWC input, KRSC weights, symmetric stride/pad."""
    name: str
    n: int
    h: int
    w: int
    c: int
    k: int          # output channels (C_out)
    r: int
    s: int
    stride: int
    pad: int
    description: str = field(default="", compare=False)

    @property
    def ho(self) -> int:
        return (self.h + 2 * self.pad - self.r) // self.stride + 1

    @property
    def wo(self) -> int:
        return (self.w + 2 * self.pad - self.s) // self.stride + 1

    @property
    def m(self) -> int:
        """GEMM rows: output pixels N*Ho*Wo."""
        return self.n * self.ho * self.wo

    @property
    def kdim(self) -> int:
        """Algorithmic GEMM depth C*R*S (no padding counted)."""
        return self.c * self.r * self.s

    @property
    def flops(self) -> int:
        """Algorithmic work, 2*M*C_out*K."""
        return 2 * self.m * self.k * self.kdim

    @property
    def compulsory_bytes(self) -> int:
        """x and W read once, y written once (bf16), scale and bias (fp32) read once."""
        return 2 * (self.n * self.h * self.w * self.c + self.k * self.r * self.s * self.c
                    + self.m * self.k) + 8 * self.k

    def with_batch(self, n: int) -> "LayerShape":
        return LayerShape(self.name, n, self.h, self.w, self.c, self.k, self.r, self.s,
                          self.stride, self.pad, self.description)


# The five YOLO-shaped layers the fused kernel is measured on.
LAYERS: dict[str, LayerShape] = {
    "tiny": LayerShape("tiny", 1, 32, 32, 16, 32, 3, 3, 1, 1,
                       "tiny correctness layer 1x32x32x16 -> 32, 3x3 s1 p1"),
    "stem": LayerShape("stem", 1, 640, 640, 3, 16, 3, 3, 2, 1,
                       "YOLO-style stem 1x640x640x3 -> 16, 3x3 s2 p1"),
    "down": LayerShape("down", 16, 160, 160, 64, 128, 3, 3, 2, 1,
                       "downsample 16x160x160x64 -> 128, 3x3 s2 p1"),
    "pointwise": LayerShape("pointwise", 16, 40, 40, 256, 256, 1, 1, 1, 0,
                            "pointwise 16x40x40x256 -> 256, 1x1 s1 p0"),
    "deep": LayerShape("deep", 32, 20, 20, 512, 512, 3, 3, 1, 1,
                       "deep 32x20x20x512 -> 512, 3x3 s1 p1"),
}
LAYER_ORDER = ("tiny", "stem", "down", "pointwise", "deep")
BASE_SEED = 0xC0B5


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns.

    Inputs are finite normal draws, so no NaN/Inf handling is needed.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class LayerInputs:
    shape: LayerShape
    x_bits: np.ndarray   # uint16 [n][h][w][c]
    w_bits: np.ndarray   # uint16 [k][r][s][c]
    gamma: np.ndarray    # float32 [k]
    beta: np.ndarray
    mean: np.ndarray
    var: np.ndarray
    eps: float


def make_layer_inputs(shape: LayerShape, seed: int | None = None) -> LayerInputs:
    """Draw one layer's inputs with the recipe in the module docstring."""
    if seed is None:
        seed = BASE_SEED + (LAYER_ORDER.index(shape.name) if shape.name in LAYER_ORDER else 0)
    streams = [np.random.Generator(np.random.PCG64(s))
               for s in np.random.SeedSequence(seed).spawn(6)]
    gx, gw, gg, gb, gm, gv = streams
    x = gx.standard_normal((shape.n, shape.h, shape.w, shape.c), dtype=np.float32)
    fan_in = shape.c * shape.r * shape.s
    w = gw.standard_normal((shape.k, shape.r, shape.s, shape.c), dtype=np.float32)
    w *= np.float32(np.sqrt(2.0 / fan_in))
    gamma = gg.uniform(0.5, 1.5, shape.k).astype(np.float32)
    beta = (gb.standard_normal(shape.k) * 0.1).astype(np.float32)
    mean = (gm.standard_normal(shape.k) * 0.1).astype(np.float32)
    var = gv.uniform(0.5, 2.0, shape.k).astype(np.float32)
    return LayerInputs(shape, f32_to_bf16_bits(x), f32_to_bf16_bits(w),
                       gamma, beta, mean, var, 1e-3)


def bits_to_torch_bf16(bits: np.ndarray):
    """View uint16 bf16 bit patterns as a CPU torch.bfloat16 tensor (no copy of values)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def torch_bf16_to_bits(t) -> np.ndarray:
    """A torch.bfloat16 tensor (any device) -> uint16 bit patterns on the host."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
