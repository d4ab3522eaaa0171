"""Pins for the oracle's e4m3 codec: bit definition, rounding, torch's cast."""

import math

import numpy as np
import pytest
import torch

from oracle import e4m3


def test_decode_spot_values_from_bit_layout():
    t = e4m3.decode_table()
    assert t[0x00] == 0.0 and not math.copysign(1.0, t[0x00]) < 0
    assert t[0x80] == 0.0 and math.copysign(1.0, t[0x80]) < 0
    assert t[0x01] == 2.0 ** -9           # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9       # largest subnormal
    assert t[0x08] == 2.0 ** -6           # smallest normal
    assert t[0x38] == 1.0                 # E=7, M=0
    assert t[0x3C] == 1.5
    assert t[0x7E] == 448.0               # largest finite
    assert t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isfinite(t).sum() == 254


def test_positive_codes_are_strictly_increasing():
    t = e4m3.decode_table()[:0x7F]
    assert np.all(np.diff(t) > 0)


def test_every_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3.decode(codes).astype(np.float32)
    np.testing.assert_array_equal(e4m3.encode(vals), codes)


def test_midpoints_round_to_even_code():
    t = e4m3.decode_table()
    for c in range(0x00, 0x7E):
        lo, hi = t[c], t[c + 1]
        mid = np.float32((lo + hi) / 2)           # exactly representable in fp32
        assert float(mid) == (lo + hi) / 2
        expect = c if c % 2 == 0 else c + 1
        assert e4m3.encode(np.array([mid]))[0] == expect, hex(c)
        assert e4m3.encode(-np.array([mid]))[0] == expect | 0x80
        # just off the midpoint goes to the nearer code
        above = np.nextafter(mid, np.float32(np.inf))
        below = np.nextafter(mid, np.float32(-np.inf))
        assert e4m3.encode(np.array([above]))[0] == c + 1
        assert e4m3.encode(np.array([below]))[0] == c


def test_saturation_and_nan():
    v = np.array([448.0, 460.0, 464.0, 465.0, 1e6, np.inf, -np.inf, -1000.0, np.nan], np.float32)
    np.testing.assert_array_equal(
        e4m3.encode(v), np.array([0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F], np.uint8))


@pytest.mark.parametrize("lo,hi", [(0.0, 2.0 ** -8), (2.0 ** -8, 1.0), (1.0, 64.0), (64.0, 464.0)])
def test_matches_torch_cpu_cast(lo, hi):
    g = np.random.default_rng(123)
    v = g.uniform(lo, hi, size=200_000).astype(np.float32)
    v = np.concatenate([v, -v])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(e4m3.encode(v), ref)


def test_golden_exact_value_list_is_every_e4m3_integer_from_1_to_64():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "e4m3_exact_values.txt")
    vals = [int(l) for l in open(path) if l.strip() and not l.startswith("#")]
    assert vals == sorted(set(vals))
    grid = e4m3.decode_table()
    exact = sorted(int(v) for v in grid[np.isfinite(grid)] if 1 <= v <= 64 and v == int(v))
    assert vals == exact
    # and each listed value survives an encode/decode round trip
    arr = np.array(vals, np.float32)
    np.testing.assert_array_equal(e4m3.decode(e4m3.encode(arr)), arr.astype(np.float64))
