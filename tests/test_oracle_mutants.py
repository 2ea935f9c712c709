"""Plants plausible mistakes in copies of the oracle and checks the pins catch each one.

Each mutant is a textual edit of the oracle's source (a wrong sign, a swapped
or transposed index, a dropped term, the stride on the wrong axis, a wrong
fold or sigmoid), compiled or imported separately on the CPU.  The test
asserts that the hand-summed fixtures, the torch float64 conv2d comparison
or the closed-form checks reject every one of them, i.e. that the oracle's
pins are strong enough to notice such a bug in the oracle itself.
"""
import ctypes
import json
import os
import subprocess
import types

import mpmath
import numpy as np
import pytest
import torch

import oracle
from conv2d_batchnorm_silu_gb300.synthetic import bf16_bits_to_f32, f32_to_bf16_bits

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_DIR = os.path.join(os.path.dirname(HERE), "oracle")

C_MUTANTS = {
    "pad_sign": ("int64_t ih = oh * p->sh - p->ph + r;", "int64_t ih = oh * p->sh + p->ph + r;"),
    "r_for_s": ("int64_t iw = ow * p->sw - p->pw + s;", "int64_t iw = ow * p->sw - p->pw + r;"),
    "kernel_flipped_true_convolution": ("((k * p->r + r) * p->s + s) * p->c",
                                        "((k * p->r + (p->r - 1 - r)) * p->s + (p->s - 1 - s)) * p->c"),
    "stride_wrong_axis": ("int64_t ih = oh * p->sh - p->ph + r;",
                          "int64_t ih = oh * p->sw - p->ph + r;"),
    "dropped_first_channel": ("for (int64_t c = 0; c < p->c; ++c) acc",
                              "for (int64_t c = 1; c < p->c; ++c) acc"),
    "batch_ignored": ("((n * p->h + ih) * p->wi + iw) * p->c", "((0 * p->h + ih) * p->wi + iw) * p->c"),
    "last_row_skipped": ("if (ih < 0 || ih >= p->h) continue;",
                         "if (ih < 0 || ih >= p->h - 1) continue;"),
}

PY_MUTANTS = {
    "bias_sign": ("bias = b - mu * scale", "bias = b + mu * scale"),
    "scale_inverted": ("scale = g / np.sqrt(v + e)", "scale = g * np.sqrt(v + e)"),
    "eps_dropped": ("scale = g / np.sqrt(v + e)", "scale = g / np.sqrt(v)"),
    "sigmoid_sign": ("return z / (1.0 + np.exp(-z))", "return z / (1.0 + np.exp(z))"),
    "plain_sigmoid": ("return z / (1.0 + np.exp(-z))", "return 1.0 / (1.0 + np.exp(-z))"),
    "bias_before_scale": ("return np.asarray(conv, dtype=np.float64) * np.asarray(scale, np.float64) \\\n        + np.asarray(bias, np.float64)",
                          "return (np.asarray(conv, dtype=np.float64) + np.asarray(bias, np.float64)) \\\n        * np.asarray(scale, np.float64)"),
    "relu_as_abs": ("return np.where(z > 0.0, z, 0.0)", "return np.abs(z)"),
    "identity_is_silu": ('if activation == "identity":\n        return np.asarray(z, dtype=np.float64)',
                         'if activation == "identity":\n        return silu(z)'),
    "residual_before_act": ("y = activate(bn(conv, scale, bias), activation)\n    if residual is not None:\n"
                            "        y = y + np.asarray(residual, dtype=np.float64)",
                            "z = bn(conv, scale, bias)\n    if residual is not None:\n"
                            "        z = z + np.asarray(residual, dtype=np.float64)\n    y = activate(z, activation)"),
    "e4m3_ties_up": ("(codes[hi] % 2 == 0) & (hi != lo)", "(hi != lo)"),
    "e4m3_sign_dropped": ("np.where(np.signbit(v), 0x80, 0)", "np.where(np.signbit(v), 0, 0)"),
}


def build_c_mutant(tmp_path, name, old, new):
    with open(os.path.join(ORACLE_DIR, "oracle.c")) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutant {name}: pattern not found"
    src = src.replace(old, new, 1)
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"lib{name}.so"
    c_path.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-ffp-contract=off", str(c_path), "-o", str(so_path), "-lm"], check=True)
    lib = ctypes.CDLL(str(so_path))
    lib.oracle_conv2d.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int64] * 11 + \
        [ctypes.c_void_p, ctypes.c_int]
    lib.oracle_conv2d.restype = ctypes.c_int
    return lib


def run_conv(lib, xb, wb, stride, pad):
    n, h, w, c = xb.shape
    k, r, s, _ = wb.shape
    ho = (h + 2 * pad[0] - r) // stride[0] + 1
    wo = (w + 2 * pad[1] - s) // stride[1] + 1
    out = np.full((n, ho, wo, k), np.nan)
    xb = np.ascontiguousarray(xb)
    wb = np.ascontiguousarray(wb)
    lib.oracle_conv2d(xb.ctypes.data, wb.ctypes.data, n, h, w, c, k, r, s,
                      stride[0], stride[1], pad[0], pad[1], out.ctypes.data, 1)
    return out


def conv_pins_pass(lib):
    """The hand fixtures and a torch float64 comparison, against library ``lib``."""
    with open(os.path.join(HERE, "golden", "conv_hand_cases.json")) as f:
        doc = json.load(f)
    for case in doc["cases"]:
        x = doc[case["x"]] if isinstance(case["x"], str) else case["x"]
        out = run_conv(lib, f32_to_bf16_bits(np.asarray(x, np.float32)),
                       f32_to_bf16_bits(np.asarray(case["w"], np.float32)),
                       case["stride"], case["pad"])
        if out.shape != np.asarray(case["expected"]).shape or \
                not np.array_equal(out, np.asarray(case["expected"], np.float64)):
            return False
    rng = np.random.default_rng(99)
    for (n, h, w, c, k, r, s, st, pd) in [(2, 9, 7, 5, 6, 3, 3, (2, 2), (1, 1)),
                                          (3, 6, 9, 2, 5, 2, 3, (1, 2), (0, 1))]:
        xb = f32_to_bf16_bits(rng.standard_normal((n, h, w, c)).astype(np.float32))
        wb = f32_to_bf16_bits(rng.standard_normal((k, r, s, c)).astype(np.float32))
        out = run_conv(lib, xb, wb, st, pd)
        xt = torch.from_numpy(bf16_bits_to_f32(xb).astype(np.float64)).permute(0, 3, 1, 2)
        wt = torch.from_numpy(bf16_bits_to_f32(wb).astype(np.float64)).permute(0, 3, 1, 2)
        ref = torch.nn.functional.conv2d(xt, wt, stride=st, padding=pd).permute(0, 2, 3, 1).numpy()
        if out.shape != ref.shape or not np.allclose(out, ref, rtol=1e-12, atol=1e-12):
            return False
    return True


def test_unmutated_oracle_passes_the_mutation_harness(tmp_path):
    lib = build_c_mutant(tmp_path, "identity", "acc = 0.0;", "acc = 0.0;")
    assert conv_pins_pass(lib)


@pytest.mark.parametrize("name", sorted(C_MUTANTS))
def test_conv_mutant_is_caught(tmp_path, name):
    old, new = C_MUTANTS[name]
    assert not conv_pins_pass(build_c_mutant(tmp_path, name, old, new))


def load_py_mutant(name, old, new):
    with open(os.path.join(ORACLE_DIR, "__init__.py")) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutant {name}: pattern not found"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    mod.__file__ = os.path.join(ORACLE_DIR, "__init__.py")
    exec(compile(src.replace(old, new, 1), mod.__file__, "exec"), mod.__dict__)
    return mod


def py_pins_pass(mod):
    mpmath.mp.dps = 50
    with open(os.path.join(HERE, "golden", "bn_fold_hand_cases.json")) as f:
        for cs in json.load(f)["cases"]:
            sc, bi = mod.bn_fold([cs["gamma"]], [cs["beta"]], [cs["mean"]], [cs["var"]], cs["eps"])
            if sc[0] != cs["scale"] or bi[0] != cs["bias"]:
                return False
    sc, bi = mod.bn_fold([1.0], [0.0], [0.0], [1.0], np.float32(1e-3))
    if abs(sc[0] - float(1 / mpmath.sqrt(1 + mpmath.mpf(float(np.float32(1e-3)))))) > 1e-15:
        return False
    for z in (-5.0, -1.0, 0.5, 3.0):
        ref = float(mpmath.mpf(z) / (1 + mpmath.exp(-mpmath.mpf(z))))
        if abs(mod.silu(z) - ref) > 1e-14:
            return False
    conv = np.array([[0.5, -1.5]])
    got = mod.bn_silu(conv, np.array([2.0, -1.0]), np.array([0.25, 1.0]))
    for k, (s, b) in enumerate([(2.0, 0.25), (-1.0, 1.0)]):
        z = conv[0, k] * s + b
        if abs(got[0, k] - float(mpmath.mpf(z) / (1 + mpmath.exp(-mpmath.mpf(z))))) > 1e-14:
            return False
    if not epilogue_pins_pass(mod):
        return False
    # fp8 e4m3 cast: a tie to even, a tie below, saturation (hand-derived in test_oracle_fp8.py)
    e = mod.to_e4m3_bits(np.array([1.0625, 17.0, 232.0, 1000.0, -1e30]))
    return [int(c) for c in e] == [0x38, 0x58, 0x76, 0x7E, 0xFE]


def epilogue_pins_pass(mod):
    """The hand-derived epilogue fixture (tests/golden/epilogue_hand_cases.json)."""
    with open(os.path.join(HERE, "golden", "epilogue_hand_cases.json")) as f:
        ep = json.load(f)
    with open(os.path.join(HERE, "golden", "conv_hand_cases.json")) as f:
        conv = json.load(f)
    case = next(c for c in conv["cases"] if c["name"] == ep["conv_case"])
    x = conv[case["x"]] if isinstance(case["x"], str) else case["x"]
    xb = f32_to_bf16_bits(np.asarray(x, np.float32))
    wb = f32_to_bf16_bits(np.asarray(case["w"], np.float32))
    for cs in ep["cases"]:
        expected = np.asarray(cs["expected"], np.float64)
        res = None
        if cs["residual"]:
            res = f32_to_bf16_bits(np.broadcast_to(np.asarray(ep["residual_per_channel"], np.float32),
                                                   expected.shape).copy())
        got = mod.conv_bn_act(xb, wb, np.float32(ep["gamma"]), np.float32(ep["beta"]), np.float32(ep["mean"]),
                              np.float32(ep["var"]), ep["eps"], case["stride"], case["pad"], cs["activation"], res,
                              threads=1)
        if got.shape != expected.shape or not np.array_equal(got, expected):
            return False
    return True


def test_unmutated_python_half_passes():
    assert py_pins_pass(oracle)


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_python_mutant_is_caught(name):
    old, new = PY_MUTANTS[name]
    assert not py_pins_pass(load_py_mutant(name, old, new))
