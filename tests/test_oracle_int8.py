"""Pins of the oracle's symmetric per-head INT8 codec ("Building a quantized
HiCache for SGLang", sections "Building the INT8 codec" and "Why exactly 1,152
bytes?"): the page's worked example and record sizes, closed forms, exhaustive
checks over BF16 maxima, exact tie cases, and an exact-rational restatement of
the FP32 quotient."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "hiq_int8.txt")


def gold():
    rows = {}
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        key, rest = line.split(None, 1)
        rows[key] = rest.split()
    return rows


def bf16(x):
    return O.bf16_to_f32(O.f32_to_bf16(np.asarray(x, np.float32)))


def test_worked_example():
    g = gold()["example"]
    arrow = g.index("->")
    vals = np.array([float(v) for v in g[:arrow]], np.float32)
    want = [int(v) for v in g[arrow + 1:]]
    for D in (32, 64, 128, 256):  # the four values padded with zeros to a head
        x = np.zeros((1, D), np.float32)
        x[0, :4] = bf16(vals)
        codes, s16 = O.int8_encode(x)
        assert list(codes[0, :4]) == want
        assert np.all(codes[0, 4:] == 0)
        assert s16[0] == 0x3C01  # BF16(fl32(1/127)) = 1.0078125 * 2^-7


def test_record_and_ratio():
    g = gold()
    r = dict(kv.split("=") for kv in g["record"])
    H, D = int(r["heads"]), int(r["head_dim"])
    assert H * D == int(r["codes"]) and 2 * H == int(r["scales"])
    assert H * D + 2 * H == int(r["raw_record"])
    assert O.int8_record_bytes(H, D) == int(r["record"]) == 9 * 128
    t = dict(kv.split("=") for kv in g["token"])
    L = int(t["layers"])
    bf = 2 * L * int(t["heads"]) * int(t["head_dim"]) * 2
    assert bf == int(t["bf16_bytes"])
    enc = 2 * L * O.int8_record_bytes(int(t["heads"]), int(t["head_dim"]))
    assert round(100 * (1 - enc / bf), 2) == float(t["reduction_percent"])
    assert round(bf / enc, 2) == float(t["capacity_x"])
    # a segment (16-token page) is 16 records
    geom = O.make_geom(dtype=O.BF16, layout=O.SEPARATE, head_dim=128, num_heads=8,
                       block_tokens=16, num_layers=1, num_blocks=1,
                       strides=(16 * 8 * 128, 8 * 128, 128), codecs=(O.INT8, O.INT8))
    assert O.segment_enc_bytes(geom, 0) == 16 * 1152
    assert O.segment_enc_bytes(geom, 0) / O.segment_raw_bytes(geom) == 0.5625


def test_record_bytes_closed_form():
    for H in range(1, 65):
        for D in (32, 64, 128, 256):
            b = O.int8_record_bytes(H, D)
            assert b % 128 == 0 and H * (D + 2) <= b < H * (D + 2) + 128


def test_scale_closed_forms():
    assert O.int8_scale(127.0) == 0x3F80          # 127 / 127 = 1
    assert O.int8_scale(127.0 * 2.0 ** -10) == 0x3A80   # 2^-10
    floor = O.int8_scale(0.0)
    assert floor == O.int8_scale(1e-13) != 0      # below the floor: the floor's scale
    assert O.bf16_to_f32(np.array([floor], np.uint16))[0] > 0


def test_all_zero_head_restores_exactly_zero():
    x = np.zeros((3, 128), np.float32)
    codes, s16 = O.int8_encode(x)
    assert np.all(codes == 0) and np.all(s16 != 0)
    assert np.all(O.int8_decode(codes, s16) == 0)


def test_max_element_codes_127_for_every_bf16_maximum():
    """Every positive finite BF16 value as the head's maximum: that element codes
    to +-127 and half of it to 64 +- 1."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint16)       # positive finite BF16
    a = O.bf16_to_f32(bits)
    a = a[a >= 1e-12]                                        # above the floor
    x = np.zeros((a.size, 32), np.float32)
    x[:, 0], x[:, 1] = a, -a
    x[:, 2] = bf16(a * 0.5)
    codes, s16 = O.int8_encode(x)
    assert np.all(codes[:, 0] == 127) and np.all(codes[:, 1] == -127)
    assert np.all(np.abs(codes[:, 2].astype(int) - 64) <= 1)
    # the rounded scale makes the quotient of the maximum exceed 127 for some
    # maxima (the page's remark), though for BF16 maxima never up to 127.5, so
    # the clamp only guards
    q = a.astype(np.float64) / O.bf16_to_f32(s16).astype(np.float64)
    assert q.max() > 127.0 and q.max() < 127.5


def test_ties_round_to_even_and_symmetry():
    """Scale exactly 2^-e (maximum 127 * 2^-e); x = (k + 1/2) 2^-e are exact
    half-way quotients: the code is the even neighbour, and -x codes to -code."""
    for e in (0, 3, 10, 40):
        k = np.arange(0, 127)
        x = np.zeros((k.size, 64), np.float32)
        x[:, 0] = 127.0 * 2.0 ** -e
        x[:, 1] = (k + 0.5) * 2.0 ** -e
        x[:, 2] = -(k + 0.5) * 2.0 ** -e
        assert np.array_equal(bf16(x), x)                   # all exact in BF16
        codes, s16 = O.int8_encode(x)
        assert np.all(O.bf16_to_f32(s16) == np.float32(2.0 ** -e))
        even = np.where(k % 2 == 0, k, k + 1)
        assert np.array_equal(codes[:, 1], even)
        assert np.array_equal(codes[:, 2], -even)


def test_power_of_two_scaling():
    rng = np.random.default_rng(3)
    x = bf16(rng.standard_normal((200, 128)).astype(np.float32))
    c0, s0 = O.int8_encode(x)
    for k in (-20, -3, 5, 30):
        c1, s1 = O.int8_encode(x * np.float32(2.0 ** k))
        assert np.array_equal(c0, c1)
        assert np.array_equal(O.bf16_to_f32(s1), O.bf16_to_f32(s0) * np.float32(2.0 ** k))


def _fl32(fr: Fraction) -> Fraction:
    """Nearest binary32 value of an exact rational (ties to even), normal range."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    m = a / ulp                      # in [2^23, 2^24)
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * lo * ulp


def _round_half_even(fr: Fraction) -> int:
    lo = fr.numerator // fr.denominator
    rem = fr - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return lo


def test_codes_against_exact_rational_quotient():
    """code = clamp(round_half_even(fl32(x / s)), -127, 127) with the FP32
    quotient formed from exact rationals; restore = code * s exactly."""
    rng = np.random.default_rng(11)
    x = bf16((rng.standard_normal((60, 32)) * np.exp(rng.standard_normal((60, 1)) * 3)).astype(np.float32))
    codes, s16 = O.int8_encode(x)
    s = O.bf16_to_f32(s16)
    back = O.int8_decode(codes, s16)
    for v in range(x.shape[0]):
        sv = Fraction(float(s[v]))
        for i in range(x.shape[1]):
            q = _fl32(Fraction(float(x[v, i])) / sv)
            want = max(-127, min(127, _round_half_even(q)))
            assert codes[v, i] == want, (v, i)
            assert Fraction(float(back[v, i])) == want * sv


def test_restore_error_bound():
    rng = np.random.default_rng(5)
    x = bf16(rng.standard_normal((500, 128)).astype(np.float32))
    codes, s16 = O.int8_encode(x)
    s = O.bf16_to_f32(s16)[:, None].astype(np.float64)
    y = O.int8_decode(codes, s16).astype(np.float64)
    amax = np.abs(x).max(axis=1, keepdims=True)
    # half a step, plus the step's own BF16 rounding carried over 127 steps
    assert np.all(np.abs(y - x) <= s / 2 + np.abs(amax - 127 * s) + 1e-30)


@pytest.mark.parametrize("H,D", [(8, 128), (3, 64), (1, 256), (5, 32)])
def test_segment_is_token_records(H, D):
    """A segment's slot is block_tokens records: [H*D int8 codes][H BF16 scales]
    [zeros to a multiple of 128]; decode restores code*scale rounded to BF16."""
    T, B = 16, 2
    rng = np.random.default_rng(H * 1000 + D)
    x = bf16(rng.standard_normal((B, T, H, D)).astype(np.float32) * 3)
    bits = O.f32_to_bf16(x)
    geom = O.make_geom(dtype=O.BF16, layout=O.SEPARATE, head_dim=D, num_heads=H, block_tokens=T,
                       num_layers=1, num_blocks=B, strides=(T * H * D, H * D, D),
                       codecs=(O.INT8, O.NONE))
    seg = O.segment_enc_bytes(geom, 0)
    rec = O.int8_record_bytes(H, D)
    if 8 * seg > 7 * T * H * D * 2:
        pytest.skip("no saving at this size: stays raw")
    descs = np.zeros(B, dtype=O.DESC_DTYPE)
    descs["block"] = np.arange(B)
    descs["enc_offset"] = np.arange(B) * seg
    enc, st = O.encode(geom, [bits, None], descs, B * seg)
    assert np.all(st == O.S_ENCODED)
    codes, s16 = O.int8_encode(x.reshape(-1, D))
    codes = codes.reshape(B, T, H, D)
    s16 = s16.reshape(B, T, H)
    for b in range(B):
        for t in range(T):
            r = enc[b * seg + t * rec: b * seg + (t + 1) * rec]
            assert np.array_equal(r[:H * D].view(np.int8).reshape(H, D), codes[b, t])
            assert np.array_equal(r[H * D:H * D + 2 * H].view(np.uint16), s16[b, t])
            assert np.all(r[H * D + 2 * H:] == 0)
    out = np.zeros_like(bits)
    res = O.decode(geom, [out, None], descs, enc, st)
    assert np.all(res == O.S_ENCODED)
    want = O.f32_to_bf16(O.int8_decode(codes.reshape(-1, D), s16.reshape(-1)))
    assert np.array_equal(out.reshape(-1, D), want)
