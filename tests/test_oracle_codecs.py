"""Pins of the oracle's codec steps against closed forms, invariants, brute force
and textbook values.

Sources: "KV precision and storage encoding" (OrbitKV), section "FP8 and
TurboQuant"; "Asymmetric KV: methods and results" (knlp), section "Precision
and scaling reference" (FP8 scale rule) and the FP32 summation bound
gamma_n = n u / (1 - n u) quoted in the same section.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
from scipy import integrate, stats

import oracle as O

HEAD_DIMS = (32, 64, 128, 256)
U32 = 2.0**-24


def gamma(n):
    return n * U32 / (1 - n * U32)


# ---------------------------------------------------------------- FP8 scale rule
def test_recip448_is_nearest_float():
    c = O.fp8_scale_from_amax(1.0)              # = fl32(1 * fl32(1/448)) = fl32(1/448)
    exact = Fraction(1, 448)
    mine = Fraction(float(c))
    for nb in (np.nextafter(c, np.float32(0)), np.nextafter(c, np.float32(1))):
        assert abs(mine - exact) < abs(Fraction(float(nb)) - exact)


def test_scale_floor_and_monotone():
    floor = O.fp8_scale_from_amax(0.0)
    assert floor == O.fp8_scale_from_amax(1e-20) == O.fp8_scale_from_amax(np.float32(1e-12))
    assert floor > 0
    a = np.sort(np.random.default_rng(0).uniform(1e-6, 448, 1000)).astype(np.float32)
    s = np.array([O.fp8_scale_from_amax(v) for v in a])
    assert np.all(np.diff(s) >= 0)
    # s = amax / 448 within two FP32 roundings
    assert np.all(np.abs(s.astype(np.float64) * 448 / a - 1) <= 2.5 * U32)


@pytest.mark.parametrize("D", HEAD_DIMS)
def test_fp8_dynamic_amax_element_codes_to_448(D):
    rng = np.random.default_rng(D)
    x = (rng.standard_normal((500, D)) * np.exp(rng.uniform(-8, 4, (500, 1)))).astype(np.float32)
    s = np.array([O.fp8_scale_from_amax(O.absmax(v)) for v in x], np.float32)
    codes = O.fp8_encode(x, s)
    j = np.argmax(np.abs(x), axis=1)
    top = codes[np.arange(len(x)), j]
    assert np.all((top & 0x7F) == 0x7E)
    assert np.all((top >> 7) == (x[np.arange(len(x)), j] < 0))


def test_fp8_all_zero_vector():
    x = np.zeros((2, 64), np.float32)
    x[1] = -0.0
    s = np.array([O.fp8_scale_from_amax(O.absmax(v)) for v in x], np.float32)
    c = O.fp8_encode(x, s)
    assert np.all(c[0] == 0x00) and np.all(c[1] == 0x80)


@pytest.mark.parametrize("D", HEAD_DIMS)
def test_fp8_error_bound(D):
    """|decode - x| <= s * (half an E4M3 step) with a few FP32 roundings: 2^-4
    relative for normals, 2^-10 * s absolute in the subnormal range."""
    rng = np.random.default_rng(7 + D)
    x = rng.standard_t(4, (400, D)).astype(np.float32)
    s = np.array([O.fp8_scale_from_amax(O.absmax(v)) for v in x], np.float32)
    codes = O.fp8_encode(x, s)
    dec = O.e4m3_to_f32(codes).astype(np.float64) * s[:, None]
    err = np.abs(dec - x)
    bound = np.maximum(np.abs(x) * 2.0**-4, s[:, None] * 2.0**-10) * (1 + 4 * U32) + 4 * U32 * np.abs(x)
    assert np.all(err <= bound)


def test_fp8_quotient_clip_and_fixed_scale():
    # a fixed scale smaller than the data needs: quotients beyond 448 clip to +-448
    x = np.array([[1000.0, -1000.0, 1.0, 0.5]], np.float32)
    c = O.fp8_encode(x, np.array([1.0], np.float32))
    assert list(c[0][:2]) == [0x7E, 0xFE]


# ---------------------------------------------------------------- random signs
def test_splitmix64_published_outputs():
    # first outputs of SplitMix64 seeded with 0, as published with the reference
    # implementation (also used to seed the xoshiro generators)
    assert O.splitmix64(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


@pytest.mark.parametrize("D", HEAD_DIMS)
def test_sign_bits_follow_the_stream(D):
    words = O.splitmix64(12345, (D + 63) // 64)
    want = np.array([(words[i // 64] >> (i % 64)) & 1 for i in range(D)], np.uint8)
    assert np.array_equal(O.signs(12345, D), want)


def test_sign_balance():
    s = np.concatenate([O.signs(seed, 256) for seed in range(200)]).astype(np.float64)
    assert abs(s.mean() - 0.5) < 4 * 0.5 / math.sqrt(s.size)


# ---------------------------------------------------------------- WHT
@pytest.mark.parametrize("D", HEAD_DIMS)
def test_wht_scale_is_nearest_float(D):
    c = O.wht_scale(D)
    r = math.isqrt(D)
    if r * r == D:
        assert Fraction(float(c)) == Fraction(1, r)
        return
    # 1/sqrt(D) is irrational; c is the nearest float iff, for both neighbours n,
    # the midpoint m of (c, n) lies on the far side of 1/sqrt(D) from c:
    # m > 1/sqrt(D)  <=>  m^2 > 1/D   (all positive)
    x = Fraction(float(c))
    for nb in (np.nextafter(c, np.float32(0)), np.nextafter(c, np.float32(1))):
        m = (x + Fraction(float(nb))) / 2
        assert (m * m > Fraction(1, D)) == (m > x)


@pytest.mark.parametrize("D", HEAD_DIMS)
def test_wht_basis_vectors_match_sylvester_closed_form(D):
    c = O.wht_scale(D)
    i = np.arange(D)
    for j in range(D):
        e = np.zeros(D, np.float32)
        e[j] = 1.0
        sign = np.array([(-1) ** bin(k & j).count("1") for k in i], np.float32)
        assert np.array_equal(O.wht(e), sign * c)


@pytest.mark.parametrize("D", HEAD_DIMS)
def test_wht_vs_fp64_matrix_and_involution(D):
    rng = np.random.default_rng(D)
    H = np.array([[(-1) ** bin(a & b).count("1") for b in range(D)] for a in range(D)], np.float64)
    assert np.array_equal(H @ H, D * np.eye(D))
    for _ in range(50):
        x = rng.standard_normal(D).astype(np.float32)
        y = O.wht(x).astype(np.float64)
        ref = H @ x.astype(np.float64) / math.sqrt(D)
        nrm = np.linalg.norm(x.astype(np.float64))
        assert np.max(np.abs(y - ref)) <= (gamma(int(math.log2(D))) + 2 * U32) * math.sqrt(D) * nrm
        assert abs(np.linalg.norm(y) / nrm - 1) < 8 * math.log2(D) * U32
        back = O.wht(O.wht(x)).astype(np.float64)
        assert np.max(np.abs(back - x)) <= 4 * math.log2(D) * U32 * nrm


# ---------------------------------------------------------------- Lloyd-Max
# J. Max, "Quantizing for minimum distortion", IRE Trans. Inf. Theory 6(1), 1960,
# Table I (normal density): outputs, and the mean squared error.
MAX_TABLE = {
    2: ([0.4528, 1.510], 0.1175),
    3: ([0.2451, 0.7560, 1.344, 2.152], 0.03455),
    4: ([0.1284, 0.3881, 0.6568, 0.9424, 1.256, 1.618, 2.069, 2.733], 0.009497),
}


def test_lloyd_max_one_bit_closed_form():
    c = O.lloyd_max_gauss(1)
    assert abs(c[1] - math.sqrt(2 / math.pi)) < 1e-14 and abs(c[0] + c[1]) < 1e-15


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_lloyd_max_matches_max_1960(bits):
    c = O.lloyd_max_gauss(bits)
    K = 1 << bits
    outs, mse_tab = MAX_TABLE[bits]
    assert np.all(np.diff(c) > 0)
    assert np.max(np.abs(c[K // 2:] - np.array(outs))) < 6e-4
    t = np.concatenate([[-np.inf], (c[1:] + c[:-1]) / 2, [np.inf]])
    mse = sum(integrate.quad(lambda x, cj=c[j]: (x - cj) ** 2 * stats.norm.pdf(x), t[j], t[j + 1],
                             epsabs=1e-14)[0] for j in range(K))
    assert abs(mse - mse_tab) / mse_tab < 2e-3


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_lloyd_max_centroid_condition_by_quadrature(bits):
    c = O.lloyd_max_gauss(bits)
    K = 1 << bits
    t = np.concatenate([[-np.inf], (c[1:] + c[:-1]) / 2, [np.inf]])
    for j in range(K):
        m1 = integrate.quad(lambda x: x * stats.norm.pdf(x), t[j], t[j + 1], epsabs=1e-15)[0]
        m0 = integrate.quad(stats.norm.pdf, t[j], t[j + 1], epsabs=1e-15)[0]
        assert abs(m1 / m0 - c[j]) < 1e-9


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("D", HEAD_DIMS)
def test_codebook_scaling_and_symmetry(bits, D):
    cent, bnd = O.codebook(bits, D)
    c = O.lloyd_max_gauss(bits)
    K = 1 << bits
    assert np.array_equal(cent, -cent[::-1])
    assert np.array_equal(bnd, -bnd[::-1]) and bnd[K // 2 - 1] == 0.0
    assert np.all(np.abs(cent.astype(np.float64) * math.sqrt(D) / c - 1) <= U32)
    mid = (c[1:] + c[:-1]) / 2
    nz = mid != 0
    assert np.all(np.abs(bnd[nz].astype(np.float64) * math.sqrt(D) / mid[nz] - 1) <= U32)
