"""Pins of the oracle's TurboQuant-K and uniform-V steps.

Source: "KV precision and storage encoding" (OrbitKV), section "FP8 and
TurboQuant": K is normalized, sign-flipped, Walsh-Hadamard rotated and coded
with Gaussian Lloyd-Max centroids; restore corrects the centroid-vector norm,
inverts the transform and applies the original FP16 norm.  V uses per-vector
uniform quantization with FP16 minimum and scale.
"""
import math

import numpy as np
import pytest

import oracle as O

HEAD_DIMS = (32, 64, 128, 256)
U32 = 2.0**-24


def sylvester(D):
    return np.array([[(-1) ** bin(a & b).count("1") for b in range(D)] for a in range(D)], np.float64)


# ---------------------------------------------------------------- centroid index
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("D", HEAD_DIMS)
def test_index_is_nearest_centroid_brute_force(bits, D):
    """Away from the boundaries the index is the nearest FP64 centroid; at each
    boundary b, y = b takes the lower index and nextafter(b, +inf) the upper."""
    c64 = O.lloyd_max_gauss(bits) / math.sqrt(D)
    cent, bnd = O.codebook(bits, D)
    rng = np.random.default_rng(bits * 1000 + D)
    y = (rng.standard_normal(200_000) / math.sqrt(D)).astype(np.float32)
    mids64 = (c64[1:] + c64[:-1]) / 2
    far = np.min(np.abs(y[:, None].astype(np.float64) - mids64[None, :]), axis=1) > 1e-6 / math.sqrt(D)
    brute = np.argmin(np.abs(y[far, None].astype(np.float64) - c64[None, :]), axis=1)
    assert np.array_equal(O.tq_index(y[far], bits, D), brute)
    # boundary behaviour, every boundary
    at = O.tq_index(bnd, bits, D)
    above = O.tq_index(np.nextafter(bnd, np.float32(np.inf)), bits, D)
    assert np.array_equal(at, np.arange(len(bnd)))
    assert np.array_equal(above, np.arange(1, len(bnd) + 1))
    # +0 and -0 both take the lower middle index
    assert list(O.tq_index(np.array([0.0, -0.0], np.float32), bits, D)) == [(1 << bits) // 2 - 1] * 2


# ---------------------------------------------------------------- TQ encode
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("D", HEAD_DIMS)
def test_tq_recovers_planted_codes(bits, D):
    """Plant codes: y* = cent[c] / |cent[c]|, x = n * diag(signs) H y* / sqrt(D)
    (FP64, the inverse of the encoder's rotation).  Encoding x must return the
    planted codes (checked against FP64 brute force) and the FP16 norm of x."""
    seed = 99 + D
    rng = np.random.default_rng(bits + D)
    c64 = O.lloyd_max_gauss(bits) / math.sqrt(D)
    H = sylvester(D) / math.sqrt(D)
    neg = O.signs(seed, D).astype(np.float64)
    sgn = 1 - 2 * neg
    K = 1 << bits
    xs, want = [], []
    for _ in range(64):
        codes = rng.integers(0, K, D)
        y = c64[codes] / np.linalg.norm(c64[codes])
        n = float(np.exp(rng.uniform(-3, 3)))
        x = (sgn * (H @ y)) * n
        xs.append(x.astype(np.float32))
        want.append(np.argmin(np.abs(y[:, None] - c64[None, :]), axis=1))
    xs = np.array(xs)
    codes, n16 = O.tq_encode(xs, bits, seed)
    assert np.array_equal(codes, np.array(want))
    n64 = np.linalg.norm(xs.astype(np.float64), axis=1)
    # FP16 norm: nearest FP16 of the FP32 norm (within one FP16 step of the FP64 one)
    nf = n16.view(np.float16).astype(np.float64)
    assert np.all(np.abs(nf - n64) <= 2.0**-10 * n64)


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("D", HEAD_DIMS)
def test_tq_decode_matches_fp64_restatement(bits, D):
    """decode = n16 * diag(signs) H (c / |c|) / sqrt(D), c = centroids of the codes."""
    seed = 5
    rng = np.random.default_rng(D * 7 + bits)
    cent, _ = O.codebook(bits, D)
    codes = rng.integers(0, 1 << bits, (50, D)).astype(np.uint8)
    n16 = np.float16(np.exp(rng.uniform(-4, 4, 50))).view(np.uint16)
    out = O.tq_decode(codes, n16, bits, seed).astype(np.float64)
    H = sylvester(D) / math.sqrt(D)
    sgn = 1 - 2 * O.signs(seed, D).astype(np.float64)
    for k in range(50):
        c = cent[codes[k]].astype(np.float64)
        ref = n16[k:k + 1].view(np.float16).astype(np.float64)[0] * sgn * (H @ (c / np.linalg.norm(c)))
        scale = np.linalg.norm(ref)
        assert np.max(np.abs(out[k] - ref)) <= (2 * math.log2(D) + 8) * U32 * scale
        # the restored vector carries the stored norm
        assert abs(np.linalg.norm(out[k]) / scale - 1) <= (2 * math.log2(D) + 8) * U32


@pytest.mark.parametrize("bits,mse", [(2, 0.1175), (3, 0.03455), (4, 0.009497)])
def test_tq_relative_error_is_lloyd_max_distortion(bits, mse):
    """On Gaussian vectors the rotated coordinates are ~N(0, 1/D); the relative
    squared error after norm correction is close to the Lloyd-Max distortion."""
    D = 128
    rng = np.random.default_rng(bits)
    x = rng.standard_normal((4000, D)).astype(np.float32)
    codes, n16 = O.tq_encode(x, bits, 3)
    out = O.tq_decode(codes, n16, bits, 3).astype(np.float64)
    rel = np.sum((out - x) ** 2, axis=1) / np.sum(x.astype(np.float64) ** 2, axis=1)
    assert abs(rel.mean() / mse - 1) < 0.1


def test_tq_zero_vector():
    x = np.zeros((2, 128), np.float32)
    x[1, :] = -0.0
    codes, n16 = O.tq_encode(x, 4, 0)
    assert np.all(codes == 7) and np.all(n16 & 0x7FFF == 0)
    out = O.tq_decode(codes, n16, 4, 0)
    assert np.all(out == 0)


# ---------------------------------------------------------------- uniform
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("D", HEAD_DIMS)
def test_uniform_bound_and_extremes(bits, D):
    rng = np.random.default_rng(bits * 10 + D)
    x = (rng.standard_normal((300, D)) * 0.5).astype(np.float32)
    codes, m16, s16 = O.uniform_encode(x, bits)
    L = (1 << bits) - 1
    m = m16.view(np.float16).astype(np.float64)
    s = s16.view(np.float16).astype(np.float64)
    x64 = x.astype(np.float64)
    mn, mx = x64.min(1), x64.max(1)
    # stored metadata: FP16 of the minimum and of the step (within one FP16 rounding)
    assert np.all(np.abs(m - mn) <= 2.0**-11 * np.abs(mn) + 2.0**-25)
    assert np.all(np.abs(s - (mx - mn) / L) <= 2.0**-11 * (mx - mn) / L * (1 + 1e-6) + 2.0**-25)
    assert np.all(codes <= L)
    j0, j1 = np.argmin(x, 1), np.argmax(x, 1)
    r = np.arange(len(x))
    assert np.all(codes[r, j0] == 0) and np.all(codes[r, j1] == L)
    dec = O.uniform_decode(codes, m16, s16).astype(np.float64)
    bound = 0.5 * s[:, None] + L * np.abs(s - (mx - mn) / L)[:, None] + np.abs(m - mn)[:, None] + 1e-6
    assert np.all(np.abs(dec - x64) <= bound)
    # away from rounding ties the code is the nearest grid point (FP64 brute force)
    q = (x64 - m[:, None]) / s[:, None]
    far = np.abs(q - np.floor(q) - 0.5) > 1e-4
    grid = np.clip(np.rint(q), 0, L)
    assert np.array_equal(codes[far], grid[far].astype(np.uint8))


def test_uniform_constant_and_zero_vectors():
    x = np.full((3, 64), 1.375, np.float32)
    x[1] = 0.0
    x[2] = -2.5
    codes, m16, s16 = O.uniform_encode(x, 4)
    assert np.all(codes == 0) and np.all(s16 == 0)
    dec = O.uniform_decode(codes, m16, s16)
    assert np.array_equal(dec, x)
    # zero extremes are stored as +0 whatever the signs of the zeros
    z = np.zeros((2, 32), np.float32)
    z[0, 5] = -0.0
    z[1, :] = -0.0
    _, mz, sz = O.uniform_encode(z, 8)
    assert np.all(mz == 0x0000) and np.all(sz == 0)
    w = np.full((1, 32), -0.0, np.float32)
    w[0, 3] = -1.0                       # maximum is a (negative) zero
    c, mw, sw = O.uniform_encode(w, 4)
    assert mw[0] == O.f32_to_f16(np.array([-1.0], np.float32))[0]
    assert sw[0] == O.f32_to_f16(np.array([1.0 / 15], np.float32))[0]


# ---------------------------------------------------------------- packing
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_pack_is_little_endian_bitstream(bits):
    rng = np.random.default_rng(bits)
    for n in (32, 64, 128, 256):
        codes = rng.integers(0, 1 << bits, n).astype(np.uint8)
        big = 0
        for i, c in enumerate(codes):
            big |= int(c) << (bits * i)
        want = np.frombuffer(big.to_bytes(n * bits // 8, "little"), np.uint8)
        packed = O.pack_bits(codes, bits)
        assert np.array_equal(packed, want)
        assert np.array_equal(O.unpack_bits(packed, n, bits), codes)
    assert list(O.pack_bits(np.array([1, 2, 3, 4], np.uint8), 4)) == [0x21, 0x43]
    if bits == 3:
        # codes 0..7 -> bits 000 100 010 110 001 101 011 111 (LSB first)
        assert list(O.pack_bits(np.arange(8, dtype=np.uint8), 3)) == [0x88, 0xC6, 0xFA]


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_uniform_fp16_metadata_overflow(bits):
    """Values beyond the FP16 range (only admitted under a bound above 65504):
    the FP16 minimum overflows to -inf.  With a finite step every quotient is
    +inf and codes as the top level; when the step overflows too, inf / inf
    is not a number and codes as the lower clamp, 0."""
    top = (1 << bits) - 1
    x = np.array([[-1e5 + i for i in range(32)],          # m = -inf, s finite
                  [-1e7 if i % 2 else 1e7 for i in range(32)]], dtype=np.float32)  # s = inf
    codes, m16, s16 = O.uniform_encode(x, bits)
    assert list(m16) == [0xFC00, 0xFC00]
    assert s16[0] not in (0x7C00, 0) and s16[1] == 0x7C00
    assert np.all(codes[0] == top) and np.all(codes[1] == 0)
