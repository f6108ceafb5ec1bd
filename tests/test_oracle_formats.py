"""Pins of the oracle's number formats against library conversions and closed forms.

FP8 rules: "KV precision and storage encoding" (OrbitKV), section "FP8 and
TurboQuant" (E4M3FN, nearest-even, signed zero, subnormals, values outside
[-448, 448] stay raw).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O

ALL16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _same_f32(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    return np.all(both_nan | (a.view(np.uint32) == b.view(np.uint32)))


def test_f16_to_f32_exhaustive_vs_numpy():
    ref = ALL16.view(np.float16).astype(np.float32)
    assert _same_f32(O.f16_to_f32(ALL16), ref)


def test_bf16_to_f32_exhaustive_vs_torch():
    ref = torch.from_numpy(ALL16.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert _same_f32(O.bf16_to_f32(ALL16), ref)


def _probe_f32(grid16_as_f32):
    """All 16-bit grid values, their midpoints and +-1..2 ulp around the midpoints,
    plus random FP32 values over the whole range."""
    g = np.sort(np.unique(grid16_as_f32[np.isfinite(grid16_as_f32)]).astype(np.float64))
    mids = ((g[1:] + g[:-1]) / 2).astype(np.float32)   # exact in FP32 (one more bit)
    pts = [g.astype(np.float32), mids]
    for k in (1, 2):
        pts.append(np.nextafter(mids, np.float32(np.inf)))
        pts.append(np.nextafter(mids, np.float32(-np.inf)))
        mids = pts[-2]
    rng = np.random.default_rng(0)
    rnd = rng.integers(0, 2**32, size=1_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    pts.append(rnd[np.isfinite(rnd)])
    return np.concatenate(pts).astype(np.float32)


def test_f32_to_f16_vs_numpy():
    x = _probe_f32(ALL16.view(np.float16).astype(np.float32))
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(O.f32_to_f16(x), ref)


def test_f32_to_bf16_vs_torch():
    grid = torch.from_numpy(ALL16.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    x = _probe_f32(grid)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16(x), ref)


# ---------------------------------------------------------------- E4M3FN
def test_e4m3_closed_form_spot_values():
    cases = [(448.0, 0x7E), (-448.0, 0xFE), (0.0, 0x00), (-0.0, 0x80), (2.0**-9, 0x01),
             (2.0**-10, 0x00),          # tie between 0 and 2^-9 -> even (0)
             (3 * 2.0**-10, 0x02),      # tie between 1 and 2 (x 2^-9) -> even (2)
             (1.0, 0x38), (17.0, 0x58), # tie 16 / 18 -> even mantissa (16)
             (19.0, 0x5A),              # tie 18 / 20 -> even mantissa (20)
             (-2.0**-12, 0x80),         # tiny negative keeps its sign
             (240.0, 0x77), (2.0**-6, 0x08)]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    got = O.f32_to_e4m3(x)
    assert [int(v) for v in got] == [c[1] for c in cases]


def test_e4m3_decode_closed_form():
    # value of every finite code from the format definition, written as rationals
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        v = O.e4m3_to_f32(np.array([c], np.uint8))[0]
        if e == 15 and m == 7:
            assert np.isnan(v)
            continue
        mag = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        assert Fraction(float(v)) == (-mag if s else mag)


def test_e4m3_exhaustive_16bit_sources_vs_torch():
    """Every finite in-range FP16 and BF16 value (the table the storage-format
    page says the GPU path is checked against), converted with scale 1."""
    for f32 in (ALL16.view(np.float16).astype(np.float32),
                torch.from_numpy(ALL16.view(np.int16).copy()).view(torch.bfloat16).float().numpy()):
        ok = np.isfinite(f32) & (np.abs(f32) <= 448)
        x = f32[ok]
        ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = O.f32_to_e4m3(x)
        assert np.array_equal(got, ref)


def test_e4m3_midpoints_and_neighbours():
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = O.e4m3_to_f32(codes).astype(np.float64)
    # round trip of every finite code, both signs
    assert np.array_equal(O.f32_to_e4m3(vals.astype(np.float32)), codes)
    assert np.array_equal(O.f32_to_e4m3(-vals.astype(np.float32)), codes | 0x80)
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    lo = codes[:-1]
    even = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(O.f32_to_e4m3(mids), even)
    assert np.array_equal(O.f32_to_e4m3(np.nextafter(mids, np.float32(0))), lo)
    assert np.array_equal(O.f32_to_e4m3(np.nextafter(mids, np.float32(np.inf))), lo + 1)
    assert np.array_equal(O.f32_to_e4m3(-mids), even | 0x80)


def test_e4m3_random_fp32_vs_torch():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(2_000_000) * np.exp(rng.uniform(-12, 6, 2_000_000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.f32_to_e4m3(x), ref)


@pytest.mark.parametrize("n", [1, 2, 4, 32, 128, 256])
def test_pairwise_sum_exact_on_integers_and_order(n):
    rng = np.random.default_rng(n)
    a = rng.integers(-1000, 1000, n).astype(np.float32)
    assert O.pairwise_sum(a) == np.float32(a.astype(np.int64).sum())
    # order pin: (1 + 2^-24) + ... lower half is summed before meeting the upper half
    if n >= 4:
        b = np.zeros(n, np.float32)
        b[0], b[1], b[n // 2] = 1.0, 2.0**-24, 2.0**-24
        # pairwise: (1 + 2^-24) rounds to 1, then + 2^-24 rounds to 1 again
        assert O.pairwise_sum(b) == np.float32(1.0)
        c = np.zeros(n, np.float32)
        c[0], c[n // 2], c[n // 2 + 1] = 1.0, 2.0**-24, 2.0**-24
        # the two small terms meet first (upper half), giving 2^-23, then 1 + 2^-23
        assert O.pairwise_sum(c) == np.float32(1.0 + 2.0**-23)
