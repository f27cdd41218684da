"""Host checks of the arithmetic the CUDA quantiser uses in place of fp32
divisions (no GPU): the scale amax/448 is computed as y0 = a*RN(1/448),
r = fma(-448, y0, a), s = fma(r, RN(1/448), y0).  For every finite bf16 value a
(group maxima are bf16) that must equal the IEEE fp32 quotient a/448, which
numpy computes here.  The FMA steps are evaluated in exact rational arithmetic
with one round-to-nearest-even to fp32 each."""
from fractions import Fraction

import numpy as np


def _rn32(fr: Fraction) -> Fraction:
    if fr == 0:
        return Fraction(0)
    neg = fr < 0
    a = -fr if neg else fr
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = a / Fraction(2) ** (e - 23)
    n, rem = divmod(q.numerator, q.denominator)
    rem = Fraction(rem, q.denominator)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = Fraction(n) * Fraction(2) ** (e - 23)
    return -v if neg else v


def test_div448_matches_ieee_for_every_bf16():
    c = np.float32(1.0) / np.float32(448.0)
    assert c.view(np.uint32) == 0x3B124925
    C = Fraction(float(c))
    bits = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    ref = bits / np.float32(448.0)
    for a, want in zip(bits.tolist(), ref):
        A = Fraction(a)
        y0 = _rn32(A * C)
        r = _rn32(A - 448 * y0)
        q = _rn32(r * C + y0)
        assert np.float32(float(q)) == want, a


def test_rn32_helper_agrees_with_numpy():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(2000) * np.exp(rng.uniform(-60, 60, 2000))
    for v in x.tolist():
        assert np.float32(float(_rn32(Fraction(v)))) == np.float32(v)



def test_fma_corrected_quotient_is_ieee_for_bf16():
    """The quantisers compute x/s as r = RN(1/s), y = RN(x*r),
    e = RN(x - s*y) (FMA), q = RN(y + e*r) (FMA), with s = fl32(amax/448).
    For bf16 x and amax, q must be the IEEE quotient fl32(x/s).  Every
    rounding commutes with scaling by powers of two (no underflow, which the
    kernels guarantee by their scale guard), so the significands of x and
    amax decide: all 128 x 128 pairs, each step in exact arithmetic with one
    rounding, x above and below amax's significand."""
    bad = []
    for am in range(128):
        amax = Fraction(128 + am, 128)
        s = _rn32(amax / 448)
        r = _rn32(1 / s)
        for xm in range(128):
            for xe in (0, -1):
                x = Fraction(128 + xm, 128) * Fraction(2) ** xe
                y = _rn32(x * r)
                e = _rn32(x - s * y)
                q = _rn32(y + e * r)
                if q != _rn32(x / s):
                    bad.append((am, xm, xe))
    assert not bad, bad[:5]


def test_fma_corrected_quotient_needs_the_correction():
    """The plain product RN(x * RN(1/s)) is not always the IEEE quotient for
    these inputs, so the correction step is doing work (a dropped FMA would
    fail the exhaustive test above)."""
    miss = 0
    for am in range(0, 128, 3):
        s = _rn32(Fraction(128 + am, 128) / 448)
        r = _rn32(1 / s)
        for xm in range(128):
            x = Fraction(128 + xm, 128)
            miss += _rn32(x * r) != _rn32(x / s)
    assert miss > 0
