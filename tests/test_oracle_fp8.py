"""Pins for the oracle's E4M3 codec (CPU only)."""
import os

import numpy as np
import pytest
import torch

from oracle import e4m3_decode, e4m3_encode

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_spec_values.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            c, v = line.split()
            rows.append((int(c, 16), float(v)))
    return rows


def test_decode_matches_spec_values():
    for code, val in _golden():
        got = e4m3_decode(np.uint8(code))
        if np.isnan(val):
            assert np.isnan(got)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)


def test_decode_all_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    mags = np.exp2(rng.uniform(-12, 8.8, size=200_000))
    x = (mags * rng.choice([-1, 1], size=mags.size)).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(x), ref)


def test_encode_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(e4m3_encode(vals), codes)


@pytest.mark.parametrize("x,code", [
    (1.0625, 0x38),        # halfway 1.0 / 1.125 -> even mantissa (1.0)
    (1.1875, 0x3A),        # halfway 1.125 / 1.25 -> 1.25
    (2.0 ** -10, 0x00),    # halfway 0 / 2^-9 -> 0
    (3 * 2.0 ** -10, 0x02),  # halfway 2^-9 / 2^-8 -> 2^-8 (even)
    (-1.0625, 0xB8),
    (464.0, 0x7E),         # beyond max: saturate
    (1e30, 0x7E),
    (float("inf"), 0x7E),
    (float("-inf"), 0xFE),
    (-1e-12, 0x80),        # rounds to zero, keeps the sign
    (float("nan"), 0x7F),
])
def test_encode_special_cases(x, code):
    assert int(e4m3_encode(np.float32(x))) == code
