"""Pins of the oracle's FP8 quotient and restore against exact rationals.

"Asymmetric KV: methods and results" (knlp), section "Precision and scaling
reference": the scale is the clamped absolute maximum times the FP32-rounded
reciprocal of 448, operands are divided in FP32, clipped to +-448 and rounded
to E4M3FN nearest/even; each layer reconstructs native operands from the codes
and FP32 scales.

Every expected value below is formed from Python Fractions, without calling the
oracle: the FP32 quotient is the binary32 value nearest the exact x / s (ties
to even), the code the E4M3FN value nearest the clipped quotient (ties to the
even fraction), and the restore the FP16 / BF16 value nearest the binary32
value nearest e4m3(code) * s.  The quotients are placed on, and one FP32 step
either side of, every midpoint between neighbouring E4M3FN values, where a
quotient off by one FP32 step changes the code; the same cases are checked to
separate the FP32 quotient from the reciprocal product x * fl32(1 / s).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from kvcases import oracle_descs

F = Fraction


# ---------------------------------------------------------------- exact rounding
def _round_binary(fr: Fraction, mant: int, emin: int) -> Fraction:
    """Nearest value with `mant` fraction bits and minimum normal exponent
    `emin` (subnormals below it), ties to the even last bit.  No overflow."""
    if fr == 0:
        return F(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    e = max(e, emin)                         # floor(log2 a), held at emin below it
    quantum = F(2) ** (e - mant)
    m = a / quantum
    n = m.numerator // m.denominator
    rem = m - n
    if rem > F(1, 2) or (rem == F(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * quantum


def fl32(fr):
    return _round_binary(F(fr), 23, -126)


def fl16(fr):
    return _round_binary(F(fr), 10, -14)


def flbf16(fr):
    return _round_binary(F(fr), 7, -126)


# E4M3FN from its definition: bias 7, 3 fraction bits, subnormals m * 2^-9,
# largest finite S.1111.110 = 448, S.1111.111 is NaN.
def _e4m3_value(c: int) -> Fraction:
    e, m = (c >> 3) & 15, c & 7
    v = F(m, 512) if e == 0 else F(8 + m) * F(2) ** (e - 10)
    return -v if c & 0x80 else v


E4M3_POS = [_e4m3_value(c) for c in range(0x7F)]          # codes 0x00 .. 0x7E, ascending
CODE_OF = {v: c for c, v in enumerate(E4M3_POS)}


def e4m3_code(q: Fraction, negative: bool) -> int:
    """Code of a quotient already clipped to [-448, 448]: 3 fraction bits with
    minimum normal exponent -6 (quantum 2^-9 below 2^-6); the sign is kept."""
    v = abs(_round_binary(q, 3, -6))
    return CODE_OF[v] | (0x80 if negative else 0)


def expected_code(x: float, s: float) -> int:
    q = fl32(F(x) / F(s))
    q = max(F(-448), min(F(448), q))
    return e4m3_code(q, np.signbit(np.float32(x)))


def dynamic_scale(amax: float) -> float:
    """s = fl32(max(amax, fl32(1e-12)) * fl32(1/448)) from exact rationals."""
    floor = fl32(F(1e-12))
    a = max(F(float(np.float32(amax))), floor)
    return float(fl32(a * fl32(F(1, 448))))


# Scales of the dynamic rule (and of fixed calibration maxima): amax values of
# every size the workloads produce, none a power of two times 448.
AMAXES = [0.013, 0.37, 1.0, 2.75, 3.9, 7.1, 19.0, 100.3, 333.0, 448.0]
SCALES = [dynamic_scale(a) for a in AMAXES]

MIDPOINTS = [(E4M3_POS[k] + E4M3_POS[k + 1]) / 2 for k in range(len(E4M3_POS) - 1)]


def _f32_neighbours(t: Fraction):
    v = np.float32(float(t))
    assert F(float(v)) == t                  # every E4M3 midpoint is a binary32 value
    return [np.nextafter(v, np.float32(-np.inf)), v, np.nextafter(v, np.float32(np.inf))]


def _dividends_for(target: np.float32, s: float):
    """FP32 dividends x whose FP32 quotient x / s is the target, or, where
    none is, the nearest quotients on both sides (found among the binary32
    values around target * s; the quotients are checked exactly later)."""
    x0 = np.float32(float(target) * s)
    cands = [x0]
    lo = hi = x0
    for _ in range(6):
        lo = np.nextafter(lo, np.float32(-np.inf))
        hi = np.nextafter(hi, np.float32(np.inf))
        cands += [lo, hi]
    t = F(float(target))
    qs = [(fl32(F(float(c)) / F(s)), c) for c in cands]
    hit = [c for q, c in qs if q == t]
    if hit:
        return hit[:1]
    below = max((qc for qc in qs if qc[0] < t), key=lambda qc: qc[0], default=None)
    above = min((qc for qc in qs if qc[0] > t), key=lambda qc: qc[0], default=None)
    return [qc[1] for qc in (below, above) if qc is not None]


def _midpoint_cases(s: float):
    xs = []
    for m in MIDPOINTS:
        for t in _f32_neighbours(m):
            xs += _dividends_for(t, s)
    xs = np.array(xs, np.float32)
    return np.concatenate([xs, -xs])


# ---------------------------------------------------------------- quotient
@pytest.mark.parametrize("s", SCALES)
def test_quotient_on_and_around_every_e4m3_midpoint(s):
    xs = _midpoint_cases(s)
    got = O.fp8_encode(xs[None, :], np.array([s], np.float32))[0]
    want = np.array([expected_code(float(x), s) for x in xs], np.uint8)
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:10]


def test_midpoint_cases_separate_quotient_from_reciprocal_product():
    """The cases above have teeth: coding x * fl32(1/s) instead of fl32(x / s)
    changes codes at most of the scales (at a power of two, here s = 1 from
    amax 448, the two agree; at some other scales the product happens to
    round like the quotient at every case)."""
    differing = 0
    for s in SCALES:
        xs = _midpoint_cases(s)
        r = np.float32(float(fl32(F(1) / F(s))))
        slip = [e4m3_code(max(F(-448), min(F(448), F(float(np.float32(x * r))))), np.signbit(x))
                for x in xs]
        want = [expected_code(float(x), s) for x in xs]
        differing += slip != want
    assert differing >= len(SCALES) // 2, differing


@pytest.mark.parametrize("s", SCALES[:4] + [1.0])
def test_quotient_of_every_fp16_value(s):
    """Every finite FP16 value as dividend (the engine's source values), with
    quotients above 448 clipped: clip + round, not rejection, here."""
    h = np.arange(0x7C00, dtype=np.uint16)
    x = O.f16_to_f32(np.concatenate([h, h | 0x8000]))
    got = O.fp8_encode(x[None, :], np.array([s], np.float32))[0]
    want = np.array([expected_code(float(v), s) for v in x], np.uint8)
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:10]
    if s < 1.0:
        assert np.any(np.abs(x / s) > 448)               # the clip is exercised
        assert np.all(got[np.abs(x.astype(np.float64) / s) > 449] & 0x7F == 0x7E)


# ---------------------------------------------------------------- segments
def _geom(codec, dtype, L=2, B=3, H=2, T=16, D=64, fixed_amax=None):
    return O.make_geom(dtype=dtype, layout=O.SEPARATE, head_dim=D, num_heads=H, block_tokens=T,
                       num_layers=L, num_blocks=B, strides=(T * H * D, H * D, D),
                       codecs=(codec, codec), fixed_amax=fixed_amax)


def _to_src(x, dtype):
    return O.f32_to_f16(x) if dtype == O.FP16 else O.f32_to_bf16(x)


def _from_src(b, dtype):
    return O.f16_to_f32(b) if dtype == O.FP16 else O.bf16_to_f32(b)


@pytest.mark.parametrize("dtype", [O.FP16, O.BF16])
@pytest.mark.parametrize("codec", [O.FP8_DYNAMIC, O.FP8_FIXED])
def test_segment_codes_and_restore_exact(codec, dtype):
    """Whole segments through the oracle's encode and decode: every code
    against the exact quotient, every restored element against the exact
    restore RN16(fl32(e4m3(c) * s)).  Fixed calibration maxima below the data's
    range make quotients beyond +-448, which clip to the largest code."""
    L, B, H, T, D = 2, 3, 2, 16, 64
    rng = np.random.default_rng(31 + codec + 7 * dtype)
    x = rng.standard_t(5, (L, 2, B, T, H, D)) * np.exp(rng.uniform(-9, 3, (L, 2, B, T, H, 1)))
    x = np.clip(x, -440, 440).astype(np.float32)
    fixed = np.array([[3.0, 0.4], [40.0, 1e-3]], np.float32)
    g = _geom(codec, dtype, L, B, H, T, D, fixed_amax=fixed if codec == O.FP8_FIXED else None)
    bits = _to_src(x, dtype)
    xs = _from_src(bits, dtype)                       # the values the codec sees
    layers = [bits[l, r].reshape(-1).copy() for l in range(L) for r in range(2)]
    seg = O.segment_enc_bytes(g, 0)
    rows = [(l, b, r, ((l * 2 + r) * B + b) * seg) for l in range(L) for r in range(2) for b in range(B)]
    enc, st = O.encode(g, layers, oracle_descs(rows), len(rows) * seg)
    assert np.all(st == O.S_ENCODED)
    nv = T * H
    clipped = 0
    for (l, b, r, off) in rows:
        v = xs[l, r, b].reshape(nv, D)
        codes = enc[off: off + nv * D].reshape(nv, D)
        if codec == O.FP8_DYNAMIC:
            s = enc[off + nv * D: off + nv * D + 4 * nv].view(np.float32)
            s_want = np.array([dynamic_scale(np.abs(row).max()) for row in v], np.float32)
            assert np.array_equal(s, s_want)
        else:
            s = np.full(nv, dynamic_scale(fixed[l, r]), np.float32)
        for i in range(nv):
            want = [expected_code(float(e), float(s[i])) for e in v[i]]
            assert list(codes[i]) == want, (l, b, r, i)
            clipped += int(np.sum(np.abs(v[i].astype(np.float64) / s[i]) > 449))
    if codec == O.FP8_FIXED:
        assert clipped > 0
    out = [np.zeros_like(a) for a in layers]
    res = O.decode(g, out, oracle_descs(rows), enc, st)
    assert np.all(res == O.S_ENCODED)
    rnd = fl16 if dtype == O.FP16 else flbf16
    for (l, b, r, off) in rows:
        codes = enc[off: off + nv * D].reshape(nv, D)
        if codec == O.FP8_DYNAMIC:
            s = enc[off + nv * D: off + nv * D + 4 * nv].view(np.float32)
        else:
            s = np.full(nv, dynamic_scale(fixed[l, r]), np.float32)
        got = _from_src(out[l * 2 + r].reshape(B, nv, D)[b], dtype)
        for i in range(nv):
            want = [rnd(fl32(_e4m3_value(int(c)) * F(float(s[i])))) for c in codes[i]]
            assert [F(float(g_)) for g_ in got[i]] == want, (l, b, r, i)


@pytest.mark.parametrize("dtype", [O.FP16, O.BF16])
def test_restore_of_every_code_exact(dtype):
    """A hand-built slot holding all 254 finite codes (and both zeros) under
    scales whose products need FP32 rounding, land in the FP16 subnormal range,
    or tie in the final 16-bit rounding: decode gives RN16(fl32(e4m3(c) * s))."""
    H, T, D = 1, 16, 32
    g = _geom(O.FP8_DYNAMIC, dtype, L=1, B=1, H=H, T=T, D=D)
    seg = O.segment_enc_bytes(g, 0)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    codes = np.resize(codes, T * D).reshape(T, D)
    codes[-1, -2:] = [0x00, 0x80]
    rng = np.random.default_rng(5)
    scales = np.concatenate([[dynamic_scale(a) for a in AMAXES[:8]],
                             [np.float32(2.0 ** -20 * 1.2345), np.float32(1.0 + 2.0 ** -8),
                              np.float32(2.0 ** -3 * (1 + 2.0 ** -9)), np.float32(7.0 / 3.0)],
                             rng.uniform(1e-4, 0.5, 4)]).astype(np.float32)
    assert scales.size == T
    slot = np.zeros(seg, np.uint8)
    slot[: T * D] = codes.reshape(-1)
    slot[T * D: T * D + 4 * T] = scales.view(np.uint8)
    out = np.zeros(T * D, np.uint16)
    res = O.decode(g, [out, np.zeros_like(out)], oracle_descs([(0, 0, 0, 0)]), slot,
                   np.array([O.S_ENCODED], np.uint8))
    assert res[0] == O.S_ENCODED
    got = _from_src(out, dtype).reshape(T, D)
    rnd = fl16 if dtype == O.FP16 else flbf16
    rounded_in_fp32 = 0
    for t in range(T):
        for d in range(D):
            exact = _e4m3_value(int(codes[t, d])) * F(float(scales[t]))
            want = rnd(fl32(exact))
            rounded_in_fp32 += fl32(exact) != exact
            assert F(float(got[t, d])) == want, (t, d, int(codes[t, d]), float(scales[t]))
            if codes[t, d] == 0x80:
                assert np.signbit(got[t, d])
    assert rounded_in_fp32 > 0


def _fp16_values_near(t: Fraction, span: int):
    """The FP16 values within `span` FP16 steps of t (t > 0 in the normal range)."""
    c = int(np.array([float(t)], np.float16).view(np.uint16)[0])
    return [float(np.array([c + k], np.uint16).view(np.float16)[0]) for k in range(-span, span + 1)]


def _boundary_cases(pred, n):
    """(calibration amax, FP16 x) pairs, found by a deterministic search over FP16
    x and FP32 scales s within three steps of x / 448 that the fixed-scale rule
    reaches (s = dynamic_scale(amax) for some FP32 amax), with pred(x, s) true."""
    r448 = fl32(F(1, 448))
    out = []
    for bits in range(0x1800, 0x5C00):          # FP16 2^-9 .. 256, increasing
        x = F(float(np.array([bits], np.uint16).view(np.float16)[0]))
        s0 = np.float32(float(x / 448))
        for k in range(-3, 4):
            sv = s0
            for _ in range(abs(k)):
                sv = np.nextafter(sv, np.float32(np.inf if k > 0 else -np.inf), dtype=np.float32)
            sf = F(float(sv))
            if not pred(x, sf):
                continue
            a0 = np.float32(float(sf / r448))
            for j in range(-4, 5):
                av = a0
                for _ in range(abs(j)):
                    av = np.nextafter(av, np.float32(np.inf if j > 0 else -np.inf), dtype=np.float32)
                if F(dynamic_scale(float(av))) == sf:
                    out.append((float(av), float(x)))
                    break
            if len(out) == n:
                return out
            break
    raise AssertionError("no boundary case found")


@pytest.mark.parametrize("mode", [0, 1])
def test_fixed_overflow_boundary(mode):
    """FP8 fixed scales and quotients beyond +-448 ("KV precision and storage
    encoding", section "FP8 and TurboQuant": values outside the range stay raw
    rather than being clipped; "Asymmetric KV", section "Precision and scaling
    reference": clipped to +-448).  Mode 0 clips (every segment encodes, the
    largest codes 0x7E / 0xFE); mode 1 keeps a segment raw exactly when one of
    its FP32 quotients fl32(x / s) lies beyond +-448.  Each segment holds one
    FP16 value within a few steps of 448 s, for scales whose quotients straddle
    the boundary, plus values where the FP32 quotient and two plausible slips
    disagree: the exact quotient (beyond 448 while fl32(x / s) = 448) and the
    product test |x| > fl32(448 s)."""
    D, T = 64, 4                                 # 4 vectors: the slot saves half the bytes
    amaxes = [0.37, 2.75, 19.0, 333.0]
    cases = []                                   # (scale index, x)
    for k, a in enumerate(amaxes):
        s = dynamic_scale(a)
        for x in _fp16_values_near(F(448) * F(s), 3):
            cases.append((k, x))
            cases.append((k, -x))
    # exact quotient beyond 448 but its FP32 value 448 (encodes), and FP32
    # quotient beyond 448 while x <= fl32(448 s) (stays raw)
    for pred in (lambda x, s: x / s > 448 and fl32(x / s) == 448,
                 lambda x, s: (fl32(x / s) > 448) != (x > fl32(448 * s))):
        for a, x in _boundary_cases(pred, 3):
            amaxes.append(a)
            cases += [(len(amaxes) - 1, x), (len(amaxes) - 1, -x)]
    B = len(cases)
    L = len(amaxes)
    fixed = np.array([[a, a] for a in amaxes], np.float32)
    g = O.make_geom(dtype=O.FP16, layout=O.SEPARATE, head_dim=D, num_heads=1, block_tokens=T,
                    num_layers=L, num_blocks=B, strides=(T * D, D, D), codecs=(O.FP8_FIXED, O.FP8_FIXED),
                    fixed_amax=fixed, fixed_overflow=mode)
    layers = []
    for l in range(L):
        for r in range(2):
            x = np.zeros((B, T, D), np.float32)
            for b, (k, v) in enumerate(cases):
                if k == l:
                    x[b, 2, 5] = v                  # token 2
                    x[b, 0, 9] = -0.5 * v            # inside the range
            layers.append(O.f32_to_f16(x.reshape(-1)))
    seg = O.segment_enc_bytes(g, 0)
    rows = [(k, b, r, (2 * b + r) * seg) for b, (k, _) in enumerate(cases) for r in range(2)]
    enc, st = O.encode(g, layers, oracle_descs(rows), len(rows) * seg)
    over = 0
    for j, (k, b, r, off) in enumerate(rows):
        s = dynamic_scale(amaxes[k])
        q = fl32(F(cases[b][1]) / F(s))
        beyond = abs(q) > 448
        over += beyond
        if mode == 1 and beyond:
            assert st[j] == O.S_RAW_RANGE, (cases[b], s, q)
        else:
            assert st[j] == O.S_ENCODED, (cases[b], s, q)
            assert enc[off + 2 * D + 5] == expected_code(cases[b][1], s)
            if beyond:
                assert enc[off + 2 * D + 5] in (0x7E, 0xFE)
    # both sides of the boundary are present, including exact quotients above
    # 448 that round to 448 in FP32 (encoded in both modes)
    assert 0 < over < len(rows)
    assert any(F(v) / F(dynamic_scale(amaxes[k])) > 448 and fl32(F(v) / F(dynamic_scale(amaxes[k]))) == 448
               for k, v in cases)
