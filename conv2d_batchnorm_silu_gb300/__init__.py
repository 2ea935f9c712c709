"""Fused conv2d -> BatchNorm -> SiLU for NVIDIA GB300 (sm_103a).

``y = SiLU(conv2d(x, W) * scale + bias)`` computed by hand-written CUDA
kernels behind the C ABI of ``include/conv_bn_silu.h``:

* ``fold``    -- BN statistics -> per-channel fp32 scale/bias;
* ``forward`` -- the fused layer on NHWC bf16 activations and KRSC bf16 weights.

The binding (``capi``) loads ``libconvbnsilu.so`` on first use and raises if
it is missing; build it with ``conv2d_batchnorm_silu_gb300._build.build()``.
``synthetic`` holds the seeded input generator and the layer shapes.
"""
from __future__ import annotations

_API = ("fold", "forward", "forward_ptr", "output_dims", "plan", "check", "CbsError", "ALGOS")


def __getattr__(name):
    if name in _API:
        from . import capi
        return getattr(capi, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")


__all__ = list(_API)
