"""Python binding of the C ABI in ``include/conv_bn_silu.h`` (ctypes).

Argument marshalling only: every step of the layer runs in the CUDA library
``libconvbnsilu.so``; this module checks tensor dtypes/layouts, passes raw
device pointers, sizes and the current CUDA stream, and turns status codes
into exceptions.  PyTorch supplies device memory and streams.  There is no
fallback: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libconvbnsilu.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
        "or conv2d_batchnorm_silu_gb300._build.build()); there is no non-CUDA fallback")

_lib = ctypes.CDLL(LIB_PATH)

CBS_OK = 0
CBS_ERR_INVALID_ARG = 1
CBS_ERR_MISALIGNED = 2
CBS_ERR_UNSUPPORTED = 3
CBS_ERR_CUDA = 4
CBS_ERR_TIMEOUT = 5

ALGOS = {"auto": 0, "tcgen05": 1, "direct": 2}
ACTIVATIONS = {"silu": 0, "identity": 1, "relu": 2}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}

_i = ctypes.c_int
_p = ctypes.c_void_p
_f = ctypes.c_float


class PlanInfo(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "algo", "block_m", "block_n", "block_k", "stages", "tiles", "grid", "threads",
        "smem_bytes", "k_iters", "stream_k", "swap_ab", "cluster")] + [("workspace_bytes", ctypes.c_longlong),
                                                                        ("balanced", ctypes.c_int),
                                                                        ("weights_resident", ctypes.c_int),
                                                                        ("row_boxes", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["algo"] = ALGO_NAMES.get(d["algo"], d["algo"])
        return d


class FoldLayer(ctypes.Structure):
    """cbs_fold_layer: one layer of conv_bn_silu_fold_batch."""
    _fields_ = [("gamma", _p), ("beta", _p), ("mean", _p), ("var", _p), ("eps", _f), ("c_out", _i),
                ("scale", _p), ("bias", _p)]


class PlanRequest(ctypes.Structure):
    """cbs_plan_request: overrides of the planner's choices (-1 / 0: planner's choice) and the
    bound on the tcgen05 kernel's pipeline waits (0: the 2 s default)."""
    _fields_ = [(name, ctypes.c_int) for name in ("algo", "swap_ab", "stream_k", "pair", "block_n")] + \
        [("wait_timeout_ns", ctypes.c_longlong), ("balanced", ctypes.c_int), ("weights_resident", ctypes.c_int),
         ("row_boxes", ctypes.c_int)]


def _request(algo="auto", swap_ab=-1, stream_k=-1, pair=-1, block_n=0, wait_timeout_ns=0,
             balanced=-1, weights_resident=-1, row_boxes=-1) -> PlanRequest:
    return PlanRequest(ALGOS[algo], int(swap_ab), int(stream_k), int(pair), int(block_n), int(wait_timeout_ns),
                       int(balanced), int(weights_resident), int(row_boxes))


def _declare(name, argtypes, restype=ctypes.c_int):
    fn = getattr(_lib, name)
    fn.argtypes = argtypes
    fn.restype = restype
    return fn


_fold = _declare("conv_bn_silu_fold", [_p, _p, _p, _p, _f, _i, _p, _p, _p])
_fold_batch = _declare("conv_bn_silu_fold_batch", [ctypes.POINTER(FoldLayer), _i, _p])
_forward = _declare("conv_bn_silu_forward", [_p] * 5 + [_i] * 11 + [_p])
_forward_algo = _declare("conv_bn_silu_forward_algo", [_p] * 5 + [_i] * 12 + [_p])
_forward_noalloc = _declare("conv_bn_silu_forward_noalloc", [_p] * 5 + [_i] * 11 + [_p])
_forward_act = _declare("conv_bn_act_forward", [_p] * 6 + [_i] * 12 + [_p])
_forward_act_fp8 = _declare("conv_bn_act_forward_fp8", [_p] * 5 + [_i] * 12 + [_p])
_forward_unfused = _declare("conv_bn_silu_forward_unfused", [_p] * 7 + [_i] * 11 + [_p])
_bn_apply = _declare("conv_bn_silu_bn_apply", [_p] * 4 + [ctypes.c_longlong, _i, _p])
_silu_apply = _declare("conv_bn_silu_silu_apply", [_p, _p, ctypes.c_longlong, _p])
_output_dims = _declare("conv_bn_silu_output_dims", [_i] * 8 + [ctypes.POINTER(_i)] * 2)
_plan = _declare("conv_bn_silu_plan", [_i] * 13 + [ctypes.POINTER(PlanInfo)])
_plan_request = _declare("conv_bn_silu_plan_request", [_i] * 11 + [ctypes.POINTER(PlanRequest), _i,
                                                                     ctypes.POINTER(PlanInfo)])
_forward_request = _declare("conv_bn_silu_forward_request", [_p] * 5 + [_i] * 11 + [ctypes.POINTER(PlanRequest), _p])
_check = _declare("conv_bn_silu_check", [_p])
_status_string = _declare("conv_bn_silu_status_string", [_i], ctypes.c_char_p)
_last_cuda_error = _declare("conv_bn_silu_last_cuda_error", [])


class CbsError(RuntimeError):
    """A non-zero cbs_status from the C library."""

    def __init__(self, status: int, what: str):
        msg = _status_string(status).decode()
        if status == CBS_ERR_CUDA:
            msg += f" (cudaError {_last_cuda_error()})"
        super().__init__(f"{what}: {msg}")
        self.status = status


def _raise_if(status: int, what: str) -> None:
    if status != CBS_OK:
        raise CbsError(status, what)


def _pair(v) -> tuple[int, int]:
    if isinstance(v, (tuple, list)):
        return int(v[0]), int(v[1])
    return int(v), int(v)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev_tensor(t: torch.Tensor, dtype: torch.dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (NHWC / KRSC dense)")
    return t.data_ptr()


def output_dims(h: int, w: int, r: int, s: int, stride=1, pad=0) -> tuple[int, int]:
    """(ho, wo) of the convolution; host only."""
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    ho, wo = _i(), _i()
    _raise_if(_output_dims(h, w, r, s, sh, sw, ph, pw, ctypes.byref(ho), ctypes.byref(wo)),
              "conv_bn_silu_output_dims")
    return ho.value, wo.value


def plan(n, h, w, c, c_out, r, s, stride=1, pad=0, algo="auto", sm_count: int = 152) -> dict:
    """The tile plan conv_bn_silu_forward_algo would use; host only."""
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    info = PlanInfo()
    _raise_if(_plan(n, h, w, c, c_out, r, s, sh, sw, ph, pw, ALGOS[algo], sm_count,
                    ctypes.byref(info)), "conv_bn_silu_plan")
    return info.as_dict()


def plan_request(n, h, w, c, c_out, r, s, stride=1, pad=0, sm_count: int = 152, **overrides) -> dict:
    """conv_bn_silu_plan_request: the plan with overrides (algo, swap_ab, stream_k, pair, block_n,
    balanced)."""
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    req = _request(**overrides)
    info = PlanInfo()
    _raise_if(_plan_request(n, h, w, c, c_out, r, s, sh, sw, ph, pw, ctypes.byref(req), sm_count,
                            ctypes.byref(info)), "conv_bn_silu_plan_request")
    return info.as_dict()


def forward_request(x: torch.Tensor, w: torch.Tensor, scale: torch.Tensor, bias: torch.Tensor,
                    stride=1, pad=0, y: torch.Tensor | None = None, stream=None, **overrides) -> torch.Tensor:
    """conv_bn_silu_forward_request: the fused forward with the planner's choices overridden."""
    n, h, wi, c = x.shape
    c_out, r, s, _ = w.shape
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    ho, wo = output_dims(h, wi, r, s, (sh, sw), (ph, pw))
    if y is None:
        y = torch.empty((n, ho, wo, c_out), dtype=torch.bfloat16, device=x.device)
    req = _request(**overrides)
    st = _forward_request(_dev_tensor(x, torch.bfloat16, "x"), _dev_tensor(w, torch.bfloat16, "w"),
                          _dev_tensor(scale, torch.float32, "scale"), _dev_tensor(bias, torch.float32, "bias"),
                          _dev_tensor(y, torch.bfloat16, "y"), n, h, wi, c, c_out, r, s, sh, sw, ph, pw,
                          ctypes.byref(req), _stream_handle(stream))
    _raise_if(st, "conv_bn_silu_forward_request")
    return y


def fold(gamma: torch.Tensor, beta: torch.Tensor, mean: torch.Tensor, var: torch.Tensor,
         eps: float, scale: torch.Tensor | None = None, bias: torch.Tensor | None = None,
         stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """conv_bn_silu_fold: per-channel fp32 scale and bias from BN statistics (device)."""
    c_out = gamma.numel()
    for t, nm in ((beta, "beta"), (mean, "mean"), (var, "var")):
        if t.numel() != c_out:
            raise ValueError(f"{nm} has {t.numel()} elements, expected {c_out}")
    if scale is None:
        scale = torch.empty(c_out, dtype=torch.float32, device=gamma.device)
    if bias is None:
        bias = torch.empty(c_out, dtype=torch.float32, device=gamma.device)
    ptrs = [_dev_tensor(t, torch.float32, nm) for t, nm in
            ((gamma, "gamma"), (beta, "beta"), (mean, "mean"), (var, "var"),
             (scale, "scale"), (bias, "bias"))]
    _raise_if(_fold(ptrs[0], ptrs[1], ptrs[2], ptrs[3], float(eps), c_out, ptrs[4], ptrs[5],
                    _stream_handle(stream)), "conv_bn_silu_fold")
    return scale, bias


class FoldBatch:
    """A prepared conv_bn_silu_fold_batch call over fixed tensors (a network's layers):
    the descriptor array is built once, each call() is one launch."""

    def __init__(self, layers):
        """layers: iterable of (gamma, beta, mean, var, eps, scale, bias); fp32 device tensors."""
        layers = list(layers)
        self._keep = layers
        self._arr = (FoldLayer * max(1, len(layers)))()
        for i, (g, b, m, v, eps, sc, bi) in enumerate(layers):
            c_out = g.numel()
            for t, nm in ((b, "beta"), (m, "mean"), (v, "var"), (sc, "scale"), (bi, "bias")):
                if t.numel() != c_out:
                    raise ValueError(f"layer {i}: {nm} has {t.numel()} elements, expected {c_out}")
            self._arr[i] = FoldLayer(_dev_tensor(g, torch.float32, "gamma"), _dev_tensor(b, torch.float32, "beta"),
                                     _dev_tensor(m, torch.float32, "mean"), _dev_tensor(v, torch.float32, "var"),
                                     float(eps), c_out, _dev_tensor(sc, torch.float32, "scale"),
                                     _dev_tensor(bi, torch.float32, "bias"))
        self._n = len(layers)

    def __call__(self, stream=None) -> None:
        _raise_if(_fold_batch(self._arr, self._n, _stream_handle(stream)), "conv_bn_silu_fold_batch")


def fold_batch(layers, stream=None) -> None:
    """conv_bn_silu_fold_batch: every layer's BN fold in one launch.

    layers: iterable of (gamma, beta, mean, var, eps, scale, bias) with fp32 device tensors;
    scale and bias are written.
    """
    FoldBatch(layers)(stream)


def forward(x: torch.Tensor, w: torch.Tensor, scale: torch.Tensor, bias: torch.Tensor,
            stride=1, pad=0, y: torch.Tensor | None = None, algo: str = "auto",
            stream=None) -> torch.Tensor:
    """conv_bn_silu_forward(_algo): y = SiLU(conv2d(x, w) * scale + bias).

    x: bf16 NHWC [n, h, w, c]; w: bf16 KRSC [c_out, r, s, c]; scale/bias: fp32 [c_out];
    y (optional, allocated if None): bf16 NHWC [n, ho, wo, c_out].
    """
    if x.dim() != 4 or w.dim() != 4:
        raise ValueError("x must be NHWC and w KRSC (4-D)")
    n, h, wi, c = x.shape
    c_out, r, s, c2 = w.shape
    if c2 != c:
        raise ValueError(f"channel mismatch: x has {c}, w has {c2}")
    if scale.numel() != c_out or bias.numel() != c_out:
        raise ValueError("scale and bias must have c_out elements")
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    ho, wo = output_dims(h, wi, r, s, (sh, sw), (ph, pw))
    if y is None:
        y = torch.empty((n, ho, wo, c_out), dtype=torch.bfloat16, device=x.device)
    elif tuple(y.shape) != (n, ho, wo, c_out):
        raise ValueError(f"y has shape {tuple(y.shape)}, expected {(n, ho, wo, c_out)}")
    if y.numel() == 0:
        return y
    px = _dev_tensor(x, torch.bfloat16, "x")
    pw_ = _dev_tensor(w, torch.bfloat16, "w")
    ps = _dev_tensor(scale, torch.float32, "scale")
    pb = _dev_tensor(bias, torch.float32, "bias")
    py = _dev_tensor(y, torch.bfloat16, "y")
    st = _forward_algo(px, pw_, ps, pb, py, n, h, wi, c, c_out, r, s, sh, sw, ph, pw,
                       ALGOS[algo], _stream_handle(stream))
    _raise_if(st, "conv_bn_silu_forward")
    return y


def forward_act(x: torch.Tensor, w: torch.Tensor, scale: torch.Tensor, bias: torch.Tensor,
                stride=1, pad=0, activation: str = "silu", residual: torch.Tensor | None = None,
                y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """conv_bn_act_forward: y = act(conv2d(x, w) * scale + bias) [+ residual].

    activation: "silu", "identity" or "relu"; residual: bf16 NHWC like y (may be y itself).
    """
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    if x.dim() != 4 or w.dim() != 4:
        raise ValueError("x must be NHWC and w KRSC (4-D)")
    n, h, wi, c = x.shape
    c_out, r, s, c2 = w.shape
    if c2 != c:
        raise ValueError(f"channel mismatch: x has {c}, w has {c2}")
    if scale.numel() != c_out or bias.numel() != c_out:
        raise ValueError("scale and bias must have c_out elements")
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    ho, wo = output_dims(h, wi, r, s, (sh, sw), (ph, pw))
    shape = (n, ho, wo, c_out)
    if y is None:
        y = torch.empty(shape, dtype=torch.bfloat16, device=x.device)
    elif tuple(y.shape) != shape:
        raise ValueError(f"y has shape {tuple(y.shape)}, expected {shape}")
    if residual is not None and tuple(residual.shape) != shape:
        raise ValueError(f"residual has shape {tuple(residual.shape)}, expected {shape}")
    if y.numel() == 0:
        return y
    pres = _dev_tensor(residual, torch.bfloat16, "residual") if residual is not None else None
    st = _forward_act(_dev_tensor(x, torch.bfloat16, "x"), _dev_tensor(w, torch.bfloat16, "w"),
                      _dev_tensor(scale, torch.float32, "scale"), _dev_tensor(bias, torch.float32, "bias"),
                      pres, _dev_tensor(y, torch.bfloat16, "y"), n, h, wi, c, c_out, r, s, sh, sw, ph, pw,
                      ACTIVATIONS[activation], _stream_handle(stream))
    _raise_if(st, "conv_bn_act_forward")
    return y


def forward_act_fp8(x: torch.Tensor, w: torch.Tensor, scale: torch.Tensor, bias: torch.Tensor,
                    stride=1, pad=0, activation: str = "silu", y: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """conv_bn_act_forward_fp8: y = act(conv2d(x, w) * scale + bias) as fp8 e4m3 bytes (torch.uint8,
    NHWC), each value rounded once to nearest even and saturated to +-448."""
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    n, h, wi, c = x.shape
    c_out, r, s, c2 = w.shape
    if c2 != c:
        raise ValueError(f"channel mismatch: x has {c}, w has {c2}")
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    ho, wo = output_dims(h, wi, r, s, (sh, sw), (ph, pw))
    shape = (n, ho, wo, c_out)
    if y is None:
        y = torch.empty(shape, dtype=torch.uint8, device=x.device)
    elif tuple(y.shape) != shape:
        raise ValueError(f"y has shape {tuple(y.shape)}, expected {shape}")
    if y.numel() == 0:
        return y
    st = _forward_act_fp8(_dev_tensor(x, torch.bfloat16, "x"), _dev_tensor(w, torch.bfloat16, "w"),
                          _dev_tensor(scale, torch.float32, "scale"), _dev_tensor(bias, torch.float32, "bias"),
                          _dev_tensor(y, torch.uint8, "y"), n, h, wi, c, c_out, r, s, sh, sw, ph, pw,
                          ACTIVATIONS[activation], _stream_handle(stream))
    _raise_if(st, "conv_bn_act_forward_fp8")
    return y


def forward_noalloc(x: torch.Tensor, w: torch.Tensor, scale: torch.Tensor, bias: torch.Tensor,
                    y: torch.Tensor, stride=1, pad=0, stream=None) -> torch.Tensor:
    """conv_bn_silu_forward_noalloc: the fused forward without any device allocation.

    For callers that must not allocate (fixed memory budgets, allocator-owned
    memory, capture-sensitive loops): the caller supplies y, and the library uses
    a fixed 20 MiB device array for its stream-K scratch.  Calls that overlap on
    the GPU share that array and race; serialise them on one stream.
    """
    if x.dim() != 4 or w.dim() != 4:
        raise ValueError("x must be NHWC and w KRSC (4-D)")
    n, h, wi, c = x.shape
    c_out, r, s, c2 = w.shape
    if c2 != c:
        raise ValueError(f"channel mismatch: x has {c}, w has {c2}")
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    ho, wo = output_dims(h, wi, r, s, (sh, sw), (ph, pw))
    if tuple(y.shape) != (n, ho, wo, c_out):
        raise ValueError(f"y has shape {tuple(y.shape)}, expected {(n, ho, wo, c_out)}")
    if y.numel() == 0:
        return y
    st = _forward_noalloc(_dev_tensor(x, torch.bfloat16, "x"), _dev_tensor(w, torch.bfloat16, "w"),
                          _dev_tensor(scale, torch.float32, "scale"),
                          _dev_tensor(bias, torch.float32, "bias"), _dev_tensor(y, torch.bfloat16, "y"),
                          n, h, wi, c, c_out, r, s, sh, sw, ph, pw, _stream_handle(stream))
    _raise_if(st, "conv_bn_silu_forward_noalloc")
    return y


def forward_unfused(x: torch.Tensor, w: torch.Tensor, scale: torch.Tensor, bias: torch.Tensor,
                    stride=1, pad=0, y: torch.Tensor | None = None, t1: torch.Tensor | None = None,
                    t2: torch.Tensor | None = None, stream=None):
    """conv_bn_silu_forward_unfused: the three-kernel sequence the fusion replaces.

    conv -> t1 (bf16), BN -> t2 (bf16), SiLU -> y (bf16); t1, t2 and y are
    allocated when not given.  Returns (y, t1, t2).  A comparator to measure
    the fused forward against, not a replacement for it.
    """
    if x.dim() != 4 or w.dim() != 4:
        raise ValueError("x must be NHWC and w KRSC (4-D)")
    n, h, wi, c = x.shape
    c_out, r, s, c2 = w.shape
    if c2 != c:
        raise ValueError(f"channel mismatch: x has {c}, w has {c2}")
    if scale.numel() != c_out or bias.numel() != c_out:
        raise ValueError("scale and bias must have c_out elements")
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    ho, wo = output_dims(h, wi, r, s, (sh, sw), (ph, pw))
    shape = (n, ho, wo, c_out)
    out = []
    for t in (y, t1, t2):
        if t is None:
            t = torch.empty(shape, dtype=torch.bfloat16, device=x.device)
        elif tuple(t.shape) != shape:
            raise ValueError(f"output has shape {tuple(t.shape)}, expected {shape}")
        out.append(t)
    y, t1, t2 = out
    if y.numel() == 0:
        return y, t1, t2
    st = _forward_unfused(_dev_tensor(x, torch.bfloat16, "x"), _dev_tensor(w, torch.bfloat16, "w"),
                          _dev_tensor(scale, torch.float32, "scale"),
                          _dev_tensor(bias, torch.float32, "bias"), _dev_tensor(t1, torch.bfloat16, "t1"),
                          _dev_tensor(t2, torch.bfloat16, "t2"), _dev_tensor(y, torch.bfloat16, "y"),
                          n, h, wi, c, c_out, r, s, sh, sw, ph, pw, _stream_handle(stream))
    _raise_if(st, "conv_bn_silu_forward_unfused")
    return y, t1, t2


def bn_apply(t1: torch.Tensor, scale: torch.Tensor, bias: torch.Tensor,
             t2: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """conv_bn_silu_bn_apply: t2 = bf16(t1 * scale[k] + bias[k]), k the innermost (channel) index."""
    c_out = scale.numel()
    if bias.numel() != c_out or t1.shape[-1] != c_out:
        raise ValueError("t1's innermost dimension, scale and bias must all have c_out elements")
    if t2 is None:
        t2 = torch.empty_like(t1)
    if t1.numel() == 0:
        return t2
    st = _bn_apply(_dev_tensor(t1, torch.bfloat16, "t1"), _dev_tensor(scale, torch.float32, "scale"),
                   _dev_tensor(bias, torch.float32, "bias"), _dev_tensor(t2, torch.bfloat16, "t2"),
                   t1.numel(), c_out, _stream_handle(stream))
    _raise_if(st, "conv_bn_silu_bn_apply")
    return t2


def silu_apply(t2: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """conv_bn_silu_silu_apply: y = bf16(SiLU(t2)), elementwise."""
    if y is None:
        y = torch.empty_like(t2)
    if t2.numel() == 0:
        return y
    st = _silu_apply(_dev_tensor(t2, torch.bfloat16, "t2"), _dev_tensor(y, torch.bfloat16, "y"),
                     t2.numel(), _stream_handle(stream))
    _raise_if(st, "conv_bn_silu_silu_apply")
    return y


def forward_ptr(x_ptr: int, w_ptr: int, scale_ptr: int, bias_ptr: int, y_ptr: int,
                n, h, w, c, c_out, r, s, stride=1, pad=0, algo: str = "auto",
                stream=None) -> None:
    """conv_bn_silu_forward_algo on raw device pointers (for callers that manage memory)."""
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    _raise_if(_forward_algo(x_ptr, w_ptr, scale_ptr, bias_ptr, y_ptr, n, h, w, c, c_out, r, s,
                            sh, sw, ph, pw, ALGOS[algo], _stream_handle(stream)),
              "conv_bn_silu_forward")


def check(stream=None) -> None:
    """conv_bn_silu_check: synchronise and raise if a kernel's pipeline wait timed out."""
    _raise_if(_check(_stream_handle(stream)), "conv_bn_silu_check")


def raw_status(fn_name: str, *args) -> int:
    """Call one C entry point with raw arguments and return its status (for tests)."""
    return getattr(_lib, fn_name)(*args)
