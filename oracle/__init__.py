"""Fp64 CPU oracle for y = SiLU(BN(conv2d(x, W))), and its other epilogues.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only code allowed to import, call or
build anything in this directory.  It shares no code with the CUDA library
and never imports it; both sides only share the seeded input generator.

Every function here is pinned by ``tests/test_oracle_*.py`` against things
fixed independently of this code (hand-summed fixtures, closed forms,
library routines, identities of the mathematics); see each docstring.

What it follows ("Fusing an Epilogue", kernels book):

* section "The problem": conv, then batch norm (a per-channel multiply and
  add), then SiLU = x * sigmoid(x);
* section "The shape of it": the convolution's accumulated result is first
  multiplied by a per-channel scale and offset by a per-channel bias, and the
  sum is then multiplied by its own sigmoid.

Readings where the page is silent (each one listed with the others in the
design notes): inference-mode BatchNorm with running statistics folded to a
per-channel scale and bias, ``scale = gamma / sqrt(var + eps)`` and
``bias = beta - mean * scale``; cross-correlation with zero padding,
dilation 1, groups 1; NHWC activations, KRSC weights, bf16 inputs decoded
exactly; all arithmetic in float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` to ``liboracle.so`` with gcc (plain C11, pthreads).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded,
    exactly as written, on x86 and on Arm alike.
    """
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64 = ctypes.c_int64
        vp = ctypes.c_void_p
        lib.oracle_conv2d.argtypes = [vp, vp] + [i64] * 11 + [vp, ctypes.c_int]
        lib.oracle_conv2d.restype = ctypes.c_int
        lib.oracle_conv2d_at.argtypes = [vp, vp] + [i64] * 11 + [vp, i64, vp, ctypes.c_int]
        lib.oracle_conv2d_at.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    """Host threads the oracle uses by default: every core this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _pair(v):
    if isinstance(v, (tuple, list)):
        return int(v[0]), int(v[1])
    return int(v), int(v)


def output_size(h: int, w: int, r: int, s: int, stride=1, pad=0) -> tuple[int, int]:
    """Output height/width of the convolution: floor((H + 2*pad - R)/stride) + 1."""
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    return (h + 2 * ph - r) // sh + 1, (w + 2 * pw - s) // sw + 1


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact decode of bf16 bit patterns (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bn_fold(gamma, beta, mean, var, eps) -> tuple[np.ndarray, np.ndarray]:
    """Fold inference BatchNorm into one multiply and one add per channel.

    BN(t) = gamma * (t - mean) / sqrt(var + eps) + beta
          = t * scale + bias, with scale = gamma / sqrt(var + eps) and
                                   bias  = beta - mean * scale.
    The fusion page treats BN as one multiply and one add with a scale and a
    bias per output channel (sections "The problem" and "The shape of it")
    but prints no fold; this is the plainest reading.  float64.
    """
    g = np.asarray(gamma, dtype=np.float64)
    b = np.asarray(beta, dtype=np.float64)
    mu = np.asarray(mean, dtype=np.float64)
    v = np.asarray(var, dtype=np.float64)
    e = np.float64(np.float32(eps)) if np.ndim(eps) == 0 else np.asarray(eps, np.float64)
    scale = g / np.sqrt(v + e)
    bias = b - mu * scale
    return scale, bias


def silu(z) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)), float64.

    ("Fusing an Epilogue", section "The problem": SiLU is x * sigmoid(x).)
    For very negative z, exp(-z) overflows to inf and the result is -0.0,
    the correctly rounded limit.
    """
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def bn(conv: np.ndarray, scale: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """Folded inference BatchNorm: z = acc*scale + bias per output channel, float64.

    ("Fusing an Epilogue", sections "The problem" and "The shape of it": batch
    norm is a multiply and an add with one scale and one bias per channel.)
    ``conv`` has output channels last; scale/bias broadcast over them.
    """
    return np.asarray(conv, dtype=np.float64) * np.asarray(scale, np.float64) \
        + np.asarray(bias, np.float64)


def bn_silu(conv: np.ndarray, scale: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """The epilogue of "The shape of it": z = acc*scale + bias, then SiLU(z)."""
    return silu(bn(conv, scale, bias))


def conv2d(x_bits: np.ndarray, w_bits: np.ndarray, stride=1, pad=0,
           threads: int | None = None) -> np.ndarray:
    """Direct convolution in float64: NHWC x (bf16 bits) with KRSC w (bf16 bits).

    out[n, ho, wo, k] = sum_{r,s,c} x[n, ho*sh - ph + r, wo*sw - pw + s, c] * w[k, r, s, c]
    with out-of-image terms dropped (zero padding).  Returns float64 NHWC.
    """
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    n, h, wi, c = x_bits.shape
    k, r, s, c2 = w_bits.shape
    if c != c2:
        raise ValueError("channel mismatch between x and w")
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    ho, wo = output_size(h, wi, r, s, (sh, sw), (ph, pw))
    out = np.empty((n, ho, wo, k), dtype=np.float64)
    rc = _load().oracle_conv2d(x_bits.ctypes.data, w_bits.ctypes.data, n, h, wi, c, k, r, s,
                               sh, sw, ph, pw, out.ctypes.data, threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_conv2d failed ({rc})")
    return out


def conv2d_at(x_bits: np.ndarray, w_bits: np.ndarray, pixels: np.ndarray, stride=1, pad=0,
              threads: int | None = None) -> np.ndarray:
    """The convolution at selected output pixels only.

    ``pixels`` holds flat output-pixel indices m = (n*Ho + ho)*Wo + wo; the
    result is float64 [len(pixels), K] (all output channels of each pixel).
    """
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    pixels = np.ascontiguousarray(pixels, dtype=np.int64)
    n, h, wi, c = x_bits.shape
    k, r, s, c2 = w_bits.shape
    if c != c2:
        raise ValueError("channel mismatch between x and w")
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    out = np.empty((pixels.size, k), dtype=np.float64)
    rc = _load().oracle_conv2d_at(x_bits.ctypes.data, w_bits.ctypes.data, n, h, wi, c, k, r, s,
                                  sh, sw, ph, pw, pixels.ctypes.data, pixels.size,
                                  out.ctypes.data, threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_conv2d_at failed ({rc})")
    return out


def conv_bn_silu(x_bits, w_bits, gamma, beta, mean, var, eps, stride=1, pad=0,
                 threads: int | None = None) -> np.ndarray:
    """The whole layer, y = SiLU(conv2d(x, W) * scale + bias), float64 NHWC."""
    scale, bias = bn_fold(gamma, beta, mean, var, eps)
    return bn_silu(conv2d(x_bits, w_bits, stride, pad, threads), scale, bias)


def conv_bn_silu_at(x_bits, w_bits, gamma, beta, mean, var, eps, pixels, stride=1, pad=0,
                    threads: int | None = None) -> np.ndarray:
    """The whole layer at selected flat output pixels: float64 [len(pixels), K]."""
    scale, bias = bn_fold(gamma, beta, mean, var, eps)
    return bn_silu(conv2d_at(x_bits, w_bits, pixels, stride, pad, threads), scale, bias)


# ---------------------------------------------------------------- other epilogues
ACTIVATIONS = ("silu", "identity", "relu")


def relu(z) -> np.ndarray:
    """max(z, 0), float64 (an activation the epilogue page names as a candidate)."""
    z = np.asarray(z, dtype=np.float64)
    return np.where(z > 0.0, z, 0.0)


def activate(z, activation: str) -> np.ndarray:
    """The activation after the BN multiply/add: "silu" (the layer), "identity" or "relu".

    ("Fusing an Epilogue", section "What an epilogue is": activations and bias
    adds are element-wise epilogue work.)
    """
    if activation == "silu":
        return silu(z)
    if activation == "identity":
        return np.asarray(z, dtype=np.float64)
    if activation == "relu":
        return relu(z)
    raise ValueError(f"unknown activation {activation!r}")


def bn_act(conv: np.ndarray, scale, bias, activation: str = "silu", residual=None) -> np.ndarray:
    """act(acc*scale + bias) [+ residual]: the residual (float64, shaped like the
    output) is added after the activation, the plainest reading of a residual
    add placed in the same epilogue."""
    y = activate(bn(conv, scale, bias), activation)
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float64)
    return y


def conv_bn_act(x_bits, w_bits, gamma, beta, mean, var, eps, stride=1, pad=0, activation: str = "silu",
                residual_bits=None, threads: int | None = None) -> np.ndarray:
    """y = act(conv2d(x, W) * scale + bias) [+ residual], float64 NHWC; residual_bits are
    bf16 bit patterns shaped like the output (decoded exactly)."""
    scale, bias = bn_fold(gamma, beta, mean, var, eps)
    res = None if residual_bits is None else bf16_bits_to_f64(residual_bits)
    return bn_act(conv2d(x_bits, w_bits, stride, pad, threads), scale, bias, activation, res)


def conv_bn_act_at(x_bits, w_bits, gamma, beta, mean, var, eps, pixels, stride=1, pad=0,
                   activation: str = "silu", residual_bits=None, threads: int | None = None) -> np.ndarray:
    """conv_bn_act at selected flat output pixels: float64 [len(pixels), K]; residual_bits
    is the full output-shaped residual, from which those pixels' rows are taken."""
    scale, bias = bn_fold(gamma, beta, mean, var, eps)
    res = None
    if residual_bits is not None:
        k = np.asarray(w_bits).shape[0]
        res = bf16_bits_to_f64(residual_bits).reshape(-1, k)[np.asarray(pixels)]
    return bn_act(conv2d_at(x_bits, w_bits, pixels, stride, pad, threads), scale, bias, activation, res)


# ---------------------------------------------------------------- fp8 e4m3 output
E4M3_MAX = 448.0


def e4m3_bits_to_f64(bits) -> np.ndarray:
    """Decode fp8 e4m3 bytes: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
    holds the subnormals m * 2^-9; 0x7f / 0xff are NaN (no infinities)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def to_e4m3_bits(values) -> np.ndarray:
    """Round float64 values to the nearest fp8 e4m3 (ties to the even mantissa), saturating
    to +-448: the narrower cast of the epilogue page's candidate list.  Written from the
    format: the representable magnitudes are enumerated and the nearest one taken."""
    v = np.asarray(values, dtype=np.float64)
    codes = np.arange(0x7F, dtype=np.uint8)                  # every non-negative finite code
    mags = e4m3_bits_to_f64(codes)                           # increasing with the code
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.clip(np.searchsorted(mags, a, side="left"), 0, len(mags) - 1)
    lo = np.clip(hi - 1, 0, len(mags) - 1)
    d_lo, d_hi = a - mags[lo], mags[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0) & (hi != lo))
    code = np.where(take_hi, codes[hi], codes[lo]).astype(np.uint8)
    code = np.where(a == mags[hi], codes[hi], code).astype(np.uint8)
    return (code | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)).astype(np.uint8)

