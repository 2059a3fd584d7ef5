"""The FP8 quantizer's quotient, restated in exact rational arithmetic (CPU).

The quantizer forms x / scale without a division per element: rc = RN(1 / scale) once per tile,
q0 = RN(x * rc), rem = RN(x - scale * q0) (a fused multiply-add: one rounding), and
q = RN(q0 + rem * rc) (another fused multiply-add), with the sign of x (the correction step of
FMA-based division, P. Markstein, IBM J. Res. Develop. 34(1), 1990).  Here every step is computed
exactly with fractions and rounded once to fp32 (round to nearest, ties to even), and the result
is compared with the correctly rounded quotient RN(x / scale): on the tile maxima and values of
every bf16 binade, near every E4M3 rounding boundary, and on random pairs.  Where |x| >= 2^-100
the two quotients must be equal; below, the exact remainder can fall under fp32's subnormal
spacing and the quotient can lose its last bit, and only the E4M3 codes (0 or -0 there: the
quotient is far below E4M3's smallest subnormal) must agree.  The GPU test
(attn_selftest_fp8_quotients) runs the kernel's own instructions over every bf16 input; this one
checks the method independently of the hardware.
"""
import random
from fractions import Fraction

import numpy as np
import pytest

from oracle import fp8 as ofp8


def rn32(v: Fraction) -> Fraction:
    """Round an exact rational to the nearest fp32 value (ties to even; normal and subnormal range,
    no overflow in these tests)."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                      # subnormals share the exponent of the smallest normal
    ulp = Fraction(2) ** (e - 23)
    m = a / ulp                           # the significand in units of the ulp
    n = m.numerator // m.denominator
    r = m - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def bf16(bits: int) -> Fraction:
    return Fraction(float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]))


def kernel_quotient(x: Fraction, sc: Fraction) -> Fraction:
    rc = rn32(1 / sc)
    q0 = rn32(x * rc)
    rem = rn32(x - sc * q0)
    q = rn32(q0 + rem * rc)
    return abs(q) if x >= 0 else -abs(q)


def scale_of(amax: Fraction) -> Fraction:
    return rn32(amax / 448)


def code(q: Fraction, negative: bool) -> int:
    v = float(q)
    if negative and v == 0.0:
        v = -0.0
    return int(ofp8.e4m3_encode(np.array([v]))[0])


def check(x_bits: int, amax_bits: int):
    x, amax = bf16(x_bits), bf16(amax_bits)
    sc = scale_of(amax)
    got, want = kernel_quotient(x, sc), rn32(x / sc)
    neg = bool(x_bits & 0x8000)
    assert code(got, neg) == code(want, neg), (hex(x_bits), hex(amax_bits))
    if abs(x) >= Fraction(2) ** -100:
        assert got == want, (hex(x_bits), hex(amax_bits))


# every binade the fast path serves (scales at or above 2^-100: amax above about 2^-91), with the
# extreme and the middle significands of the tile maximum
AMAX = [(e << 7) | m for e in range(40, 255, 3) for m in (0x00, 0x01, 0x2A, 0x40, 0x55, 0x7F)]


@pytest.mark.parametrize("amax_bits", AMAX[::7])
def test_quotient_on_the_whole_range_of_one_tile(amax_bits):
    # x = amax itself, its neighbours, and a spread of values down the binades below it
    xs = {amax_bits, max(amax_bits - 1, 0), 0, 1}
    xs |= {max(amax_bits - (k << 7) - d, 0) for k in range(0, 20) for d in (0, 1, 63, 64, 127)}
    for xb in xs:
        check(xb, amax_bits)
        check(xb | 0x8000, amax_bits)


def test_quotient_near_e4m3_rounding_boundaries():
    # x / scale lands on or next to a midpoint between E4M3 values when x = midpoint * scale is a
    # bf16 number: tiles whose maximum is 448 * 2^k (scale 2^k exactly) and 7 * 2^k (scale 2^k / 64)
    amaxes = [0x43E0 + (k << 7) for k in range(-60, 60)] + [0x40E0 + (k << 7) for k in range(-60, 60)]
    mids = [Fraction(2 * m + 1, 16) * Fraction(2) ** e for m in range(8, 16) for e in range(-9, 9)]
    for ab in amaxes:
        sc = scale_of(bf16(ab))
        for mid in mids:
            target = mid * sc
            # the bf16 values around x = midpoint * scale
            f = float(target)
            b = int(np.array([f], dtype=np.float32).view(np.uint32)[0]) >> 16
            for xb in (b - 1, b, b + 1):
                if 0 <= xb <= ab:
                    check(xb, ab)


def test_quotient_on_random_pairs():
    rnd = random.Random(20260007)
    for _ in range(2000):
        ab = rnd.randrange(0x2280, 0x7F80)          # amax from about 2^-58 up to the largest finite
        xb = rnd.randrange(0, ab + 1)
        check(xb, ab)
        check(xb | 0x8000, ab)


def test_rn32_agrees_with_float32_conversion():
    # the rounding helper itself, against numpy's float32 rounding of values exact in float64
    rnd = random.Random(7)
    for _ in range(2000):
        v = rnd.uniform(-1e6, 1e6) * 2.0 ** rnd.randrange(-60, 60)
        assert rn32(Fraction(v)) == Fraction(float(np.float32(v)))
