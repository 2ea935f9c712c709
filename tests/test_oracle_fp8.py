"""Pins for the oracle's fp8 e4m3 cast (CPU only): the narrower output cast
("Fusing an Epilogue", section "What an epilogue is").  e4m3: 1 sign bit, 4
exponent bits with bias 7, 3 mantissa bits, subnormals m * 2^-9, largest finite
448, no infinities.  Pinned by hand-derived values (ties to even at every kind
of boundary, subnormals, saturation), by an independent library conversion
(torch.float8_e4m3fn) on in-range values, and by the decode/encode round trip
of every finite code.
"""
import numpy as np
import pytest
import torch

import oracle

HAND = [
    # value, expected code, why
    (0.0, 0x00, "zero"),
    (1.0, 0x38, "exponent 7 (bias), mantissa 0"),
    (-1.0, 0xB8, "sign bit"),
    (448.0, 0x7E, "largest finite: exponent 15, mantissa 6"),
    (1000.0, 0x7E, "saturates to 448"),
    (-1e30, 0xFE, "saturates to -448"),
    (2.0 ** -9, 0x01, "smallest subnormal"),
    (2.0 ** -10, 0x00, "tie between 0 and 2^-9: even (0)"),
    (3 * 2.0 ** -10, 0x02, "tie between 2^-9 and 2*2^-9: even (2)"),
    (1.0625, 0x38, "tie between 1 and 1.125: even mantissa 0"),
    (1.1875, 0x3A, "tie between 1.125 and 1.25: even mantissa 2"),
    (232.0, 0x76, "tie between 224 and 240: even mantissa 6"),
    (17.0, 0x58, "tie between 16 and 18: even mantissa 0"),
    (17.01, 0x59, "just above the tie: 18"),
    (0.3, 0x2A, "nearest of 0.28125 and 0.3125"),
    (7 * 2.0 ** -9, 0x07, "largest subnormal"),
    (2.0 ** -6, 0x08, "smallest normal"),
]


@pytest.mark.parametrize("value,code,why", HAND, ids=[h[2] for h in HAND])
def test_hand_values(value, code, why):
    assert int(oracle.to_e4m3_bits(np.array([value]))[0]) == code, why


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_bits_to_f64(codes)
    back = oracle.to_e4m3_bits(vals)
    nonzero = vals != 0
    assert np.array_equal(back[nonzero], codes[nonzero])
    assert np.all(np.diff(oracle.e4m3_bits_to_f64(np.arange(0x7F, dtype=np.uint8))) > 0)  # increasing


def test_matches_torch_float8_on_in_range_values():
    rng = np.random.default_rng(0)
    v = np.clip(np.concatenate([rng.normal(0, 30, 50000), rng.normal(0, 0.01, 50000)]), -448, 448)
    v = v.astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = oracle.to_e4m3_bits(v.astype(np.float64))
    nz = v != 0
    assert np.array_equal(ours[nz], ref[nz])


def test_relative_error_bound():
    rng = np.random.default_rng(1)
    v = rng.uniform(2.0 ** -6, 448, 20000) * rng.choice([-1, 1], 20000)
    d = oracle.e4m3_bits_to_f64(oracle.to_e4m3_bits(v))
    assert np.all(np.abs(d - v) <= 2.0 ** -4 * np.abs(v))
