"""Pins for the oracle's element decoding and fp16 rounding (CPU only).

Each check compares the oracle with something other than itself: the
closed-form E2M1 value set of the OCP MX FP4 format, torch's float8_e4m3fn
conversion (a library routine) and numpy's float64 -> float16 cast.
"""
import math

import numpy as np
import pytest
import torch

import oracle

# OCP Microscaling Formats v1.0, FP4 E2M1: the eight magnitudes of codes 0..7.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_table_matches_format_value_set():
    t = oracle.e2m1_table()
    assert t.shape == (16,)
    for code in range(8):
        assert t[code] == E2M1_MAGNITUDES[code]
        assert not math.copysign(1.0, t[code]) < 0
        assert t[code + 8] == -E2M1_MAGNITUDES[code]
    # code 0x8 is negative zero, not a NaN or a distinct value
    assert t[8] == 0.0 and math.copysign(1.0, t[8]) < 0
    assert np.all(np.isfinite(t))


def test_e4m3_table_matches_torch_float8_e4m3fn():
    t = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_t, nan_r = np.isnan(t), np.isnan(ref)
    assert np.array_equal(nan_t, nan_r)
    assert np.array_equal(np.nonzero(nan_t)[0], [0x7F, 0xFF])
    assert np.array_equal(t[~nan_t], ref[~nan_r])
    assert np.array_equal(np.signbit(t[~nan_t]), np.signbit(ref[~nan_r]))


@pytest.mark.parametrize("code,value", [(0x38, 1.0), (0x40, 2.0), (0x48, 4.0), (0x30, 0.5),
                                        (0x28, 0.25), (0x7E, 448.0), (0x01, 2.0 ** -9),
                                        (0x18, 1 / 16), (0x24, 3 / 16), (0x70, 128.0),
                                        (0xB8, -1.0), (0x80, -0.0)])
def test_e4m3_spot_values(code, value):
    assert oracle.e4m3_table()[code] == value


def _np_half_bits(x):
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def test_fp16_rne_matches_numpy_on_random_doubles():
    rng = np.random.default_rng(1)
    mant = rng.uniform(-1, 1, 200000)
    expo = rng.integers(-30, 18, 200000)
    x = np.ldexp(mant, expo)
    assert np.array_equal(oracle.fp16_rne(x), _np_half_bits(x))


def test_fp16_rne_ties_and_edges():
    # every midpoint between consecutive finite positive halves, and both neighbours
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2.0
    for x in (h, mids, -h, -mids):
        assert np.array_equal(oracle.fp16_rne(x), _np_half_bits(x))
    special = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, np.inf, -np.inf,
                        2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26, 2.0 ** -14])
    assert np.array_equal(oracle.fp16_rne(special), _np_half_bits(special))
    assert oracle.fp16_rne([np.nan])[0] & 0x7C00 == 0x7C00 and oracle.fp16_rne([np.nan])[0] & 0x3FF


def test_fp16_from_scaled_int_matches_numpy():
    rng = np.random.default_rng(2)
    vals = []
    for bits in range(1, 53):
        vals.extend(int(v) for v in rng.integers(-(1 << bits), 1 << bits, 40))
    # exact ties: odd multiples of half a quantum, for several exponents
    for e in range(-14, 16):
        q = 2.0 ** (e - 10)
        for j in (1, 3, 5, 2047, 2049):
            v = (2.0 ** e) + (j * q / 2.0)
            n = v * 2.0 ** 20
            if n == int(n) and abs(n) < 2 ** 53:
                vals.extend([int(n), -int(n)])
    for n in vals:
        x = float(n) * 2.0 ** -20  # exact: |n| < 2^53
        assert oracle.fp16_from_scaled_int(n) == int(_np_half_bits([x])[0]), n
