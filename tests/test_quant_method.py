"""CPU checks of the arithmetic the quantiser kernels use for the codes.

The kernels compute rne(RN(x / s)) for fp16 x and a normal fp16 scale s
without dividing: t1 = RN(x * RN(1 / s)), the residual e = RN(x - t1 s) and
t2 = RN(t1 + e * RN(1 / s)) (two fused multiply-adds), then rne(t2).  That
rests on a property of fp16 quotients -- x / s is a half-integer or at least
2**-12 away from every one -- checked here, and the steps are replayed with
exact rationals and correct fp32 rounding against the definition, ties
included.  Neither the library nor the oracle is involved.
"""

from fractions import Fraction

import numpy as np

F16_FINITE = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)   # every finite fp16 >= 0


def _normal_scales(rng, n):
    bits = rng.integers(0x0400, 0x5800, size=n).astype(np.uint16)       # normal fp16 up to 128
    return bits.view(np.float16)


def test_fp16_quotients_avoid_half_integers():
    """x / s is a half-integer or at least 2**-12 away from every one
    (|x / s| <= 127.07, s a normal fp16; exact integer arithmetic)."""
    rng = np.random.default_rng(0)
    X = np.round(F16_FINITE.astype(np.float64) * 2.0 ** 24).astype(np.int64)    # x = X * 2**-24 exactly
    worst = 1.0
    scales = np.concatenate([_normal_scales(rng, 300), np.array([2.0 ** -14, 2.0 ** -6, 1.0], np.float16)])
    for s in scales:
        S = int(round(float(s) * 2 ** 24))
        xs = X[X <= int(127.07 * S)]
        two = 2 * xs
        fl = two // S
        odd = np.where(fl % 2 == 0, fl + 1, fl)
        dist = np.minimum(np.abs(two - odd * S), np.abs(two - (odd - 2) * S))   # |2x - (2k+1) s| in units
        nz = dist[dist > 0]
        if nz.size:
            worst = min(worst, nz.min() / (2 * S))
    assert worst >= 2.0 ** -12


def _rn32(q):
    """q rounded to the nearest fp32 (ties to even), q a Fraction in the normal range or 0."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    n = a / ulp
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def _rne(q):
    fl = q.numerator // q.denominator
    rem = q - fl
    return fl + (1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1) else 0)


def test_division_free_codes_match_the_definition():
    rng = np.random.default_rng(1)
    checked = ties = 0
    for sb in rng.integers(0x0400, 0x5800, size=150):
        s = Fraction(float(np.uint16(sb).view(np.float16)))
        rcp = _rn32(1 / s)
        for d in (127, 7, 1):
            xs = [Fraction(float(v)) for v in (rng.uniform(-1, 1, 30) * float(s) * d).astype(np.float16)]
            for j in rng.integers(-d, d, 12):                 # exact ties x / s = j + 1/2
                h = (int(j) + Fraction(1, 2)) * s
                if Fraction(float(np.float16(float(h)))) == h:
                    xs.append(h)
                    ties += 1
            for x in xs:
                if abs(x / s) > d * Fraction(10011, 10000):
                    continue
                t1 = _rn32(x * rcp)
                e = _rn32(x - t1 * s)
                t2 = _rn32(t1 + e * rcp)
                assert _rne(t2) == _rne(_rn32(x / s)), (float(x), float(s))
                checked += 1
    assert ties > 100 and checked > 10000
