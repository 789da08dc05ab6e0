"""The GPU kernels form each group's scale s = amax / 448 without a full IEEE
division: with y = RN(1/448), q0 = RN(amax * y), r = amax - q0 * 448 (exact
in one FMA) and s = RN(q0 + r * y) (one FMA), the correction step of
Markstein's division method.  These tests check, with exact integer and
rational arithmetic, that s equals the correctly rounded quotient: for every
fp32 amax of one binade (the step commutes with powers of two while every
intermediate stays normal) and for samples across the binades the kernels
use it for (amax >= 2**-96; smaller amax takes the IEEE division)."""

from fractions import Fraction

import numpy as np

Y = np.float32(1.0) / np.float32(448.0)        # RN(1/448), IEEE fp32 division


def _rne_shift(n, shift):
    """round(n / 2**shift), ties to even, for int64 n >= 0."""
    q = n >> shift
    rem = n - (q << shift)
    half = np.int64(1) << (shift - 1)
    up = (rem > half) | ((rem == half) & ((q & 1) == 1))
    return q + up.astype(np.int64)


def _rne_fraction_to_f32(x: Fraction) -> Fraction:
    """Correctly rounded fp32 of a positive rational in the normal range."""
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    q, r = divmod(x, ulp)
    q = int(q)
    if r * 2 > ulp or (r * 2 == ulp and q % 2 == 1):
        q += 1
    return q * ulp


def test_correction_step_is_exact_over_a_binade():
    m, e = np.frexp(np.float64(Y))
    yi, ey = int(m * 2 ** 24), int(e) - 24                 # Y = yi * 2**ey exactly
    M = np.arange(2 ** 23, 2 ** 24, dtype=np.int64)        # amax = M * 2**-23 in [1, 2)
    # Quotients lie in [2**-9, 2**-7): work in units of 2**-32 (the ulp of the
    # lower binade); a result of 2**24 units or more has ulp 2**-31.
    def to_f32_units(total, shift):
        q = _rne_shift(total, shift)
        return np.where(q >= 2 ** 24, _rne_shift(total, shift + 1) * 2, q)
    want = (M * 8) // 7
    rem = M * 8 - 7 * want
    want = want + ((2 * rem > 7) | ((2 * rem == 7) & (want % 2 == 1)))
    coarse = (M * 4) // 7
    rem = M * 4 - 7 * coarse
    coarse = (coarse + ((2 * rem > 7) | ((2 * rem == 7) & (coarse % 2 == 1)))) * 2
    want = np.where(M * 8 >= 7 * 2 ** 24, coarse, want)
    q0 = to_f32_units(M * yi, -(-23 + ey + 32))            # RN(amax * y)
    r = M * 512 - q0 * 448                                 # amax - q0*448, exact
    s = to_f32_units(q0 * (1 << -ey) + r * yi, -ey)        # RN(q0 + r*y), one rounding
    assert np.array_equal(s, want)


def test_correction_step_is_exact_across_binades():
    rng = np.random.default_rng(0)
    y = Fraction(float(Y))
    for _ in range(3000):
        a = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** int(rng.integers(-96, 100)))
        A = Fraction(float(a))
        q0 = _rne_fraction_to_f32(A * y)
        r = A - q0 * 448
        assert r == 0 or _rne_fraction_to_f32(abs(r)) == abs(r)   # the FMA's result is exact
        s = _rne_fraction_to_f32(q0 + r * y)
        assert s == _rne_fraction_to_f32(A / 448)
