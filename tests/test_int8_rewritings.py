"""Exact rewritings of the INT8 per-head encoder, checked exhaustively on the
CPU over every value they can meet (BF16 head maxima at or above the floor):

* the scale quotient a / 127 as q0 = RN(a * RN(1/127)), e = RN(fma(-q0, 127, a)),
  RN(fma(e, RN(1/127), q0)) equals the IEEE FP32 quotient;
* the clamp to [-127, 127] never acts: the FP32 quotient of the maximum by its
  BF16 scale stays below 127.5, and smaller |x| give smaller quotients.

Exact rational arithmetic (fractions) stands in for the single roundings."""
from fractions import Fraction

import numpy as np

import oracle as O


def _rn32(fr: Fraction) -> Fraction:
    """Nearest binary32 value of a positive rational in the normal range, ties to even."""
    e = fr.numerator.bit_length() - fr.denominator.bit_length()
    if Fraction(2) ** e > fr:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    m = fr / ulp
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return lo * ulp


def _maxima():
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint16)       # positive finite BF16
    a = O.bf16_to_f32(bits)
    floor = O.bf16_to_f32(O.f32_to_bf16(np.array([1e-12], np.float32)))[0]
    return np.unique(np.where(a < np.float32(1e-12), floor, a))


def test_div127_by_reciprocal_and_one_fma_is_exact():
    r = _rn32(Fraction(1, 127))
    assert r == Fraction(float(np.float32(1.0) / np.float32(127.0)))
    for a in _maxima():
        a = Fraction(float(a))
        q0 = _rn32(a * r)
        e = a - q0 * 127                       # the FMA's exact residual ...
        if e != 0:
            e = (_rn32(abs(e)) if e > 0 else -_rn32(-e))   # ... rounded once
        got = _rn32(q0 + e * r)
        assert got == _rn32(a / 127), float(a)


def test_clamp_never_acts_for_bf16_sources():
    a = _maxima()
    x = np.zeros((a.size, 32), np.float32)
    x[:, 0] = a
    _, s16 = O.int8_encode(x)
    s = O.bf16_to_f32(s16)
    q = np.array([_rn32(Fraction(float(ai)) / Fraction(float(si))) for ai, si in zip(a, s)])
    assert max(q) < Fraction(255, 2)
