"""Pins of the oracle's E4M3 codec (OCP 8-bit float, E4M3 variant).

The codec is checked against torch's independent float8_e4m3fn conversion, the
values the OCP format fixes (max 448, smallest subnormal 2^-9, NaN = 0x7F), an
exhaustive round trip, ties-to-even at every midpoint and saturation."""
import math

import numpy as np
import pytest
import torch


def test_spec_values(oracle_mod):
    d = oracle_mod.e4m3_decode
    assert d(0x00) == 0.0
    assert d(0x01) == 2.0 ** -9            # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9        # largest subnormal
    assert d(0x08) == 2.0 ** -6            # smallest normal
    assert d(0x38) == 1.0                  # exponent field 7 = bias
    assert d(0x7E) == 448.0                # largest finite
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    assert d(0xFE) == -448.0
    assert d(0x80) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0


def test_decode_matches_torch_exhaustive(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle_mod.e4m3_decode_all()
    both_nan = np.isnan(ref) & np.isnan(mine)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    assert np.array_equal(ref[~both_nan], mine[~both_nan])


def test_round_trip_all_finite_codes(oracle_mod):
    for c in range(256):
        v = oracle_mod.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert oracle_mod.e4m3_encode(v) == c, hex(c)


def test_ties_to_even_at_every_midpoint(oracle_mod):
    for c in range(0x00, 0x7E):
        lo, hi = oracle_mod.e4m3_decode(c), oracle_mod.e4m3_decode(c + 1)
        mid = 0.5 * (lo + hi)
        even = c if (c & 1) == 0 else c + 1
        assert oracle_mod.e4m3_encode(mid) == even, hex(c)
        assert oracle_mod.e4m3_encode(-mid) == (even | 0x80), hex(c)
        # just off the midpoint goes to the nearer neighbour
        assert oracle_mod.e4m3_encode(np.nextafter(mid, lo)) == c
        assert oracle_mod.e4m3_encode(np.nextafter(mid, hi)) == c + 1


def test_saturation(oracle_mod):
    enc = oracle_mod.e4m3_encode
    for x in (448.0, 448.5, 463.9, 464.0, 480.0, 1e6, float("inf")):
        assert enc(x) == 0x7E
        assert enc(-x) == 0xFE
    assert enc(float("nan")) == 0x7F


def test_agrees_with_torch_in_range(oracle_mod):
    g = torch.Generator().manual_seed(7)
    x = torch.cat([
        (torch.rand(20000, generator=g) * 2 - 1) * 448,
        torch.randn(20000, generator=g) * 0.05,
        torch.randn(20000, generator=g) * 4e-3,
    ]).to(torch.float32)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle_mod.e4m3_encode(float(v)) for v in x.numpy()], dtype=np.uint8)
    assert np.array_equal(ref, mine)
