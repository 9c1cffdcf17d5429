"""The quantiser divides each value by its block scale with Markstein's
refinement (P. Markstein, "Computation of elementary functions on the IBM
RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990) instead of an
IEEE division: from y = RN(1/b), q = RN(a y), then twice r = a - q b (one
fma) and q = RN(q + r y).  This checks, in exact rational arithmetic, that
the result is the correctly rounded fp32 quotient over the range the kernel
uses it in (2^-60 <= b <= 2^60, b = RN(amax / 448), |a| <= amax), so that
codes stay bit-identical to the oracle's IEEE division.  Quotients of at
most 2^-10 in magnitude round to a zero e4m3 code whatever their last bits,
so they are not required to match."""
import random
from fractions import Fraction as F


def rn32(x: F) -> F:
    """x rounded to the nearest fp32 value, ties to even (no overflow)."""
    if x == 0:
        return F(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    if F(2) ** (e + 1) <= a:
        e += 1
    ulp = F(2) ** (max(e, -126) - 23)
    m = a / ulp
    lo = m.numerator // m.denominator
    rest = m - lo
    if rest > F(1, 2) or (rest == F(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * lo * ulp


def markstein(a: F, b: F, y: F) -> F:
    q = rn32(a * y)
    for _ in range(2):
        r = rn32(a - q * b)  # fma: exact product, one rounding
        q = rn32(q + r * y)  # fma
    return q


def _cases(n, seed):
    rng = random.Random(seed)
    for _ in range(n):
        e = rng.choice([-60, 59]) if rng.random() < 0.1 else rng.randint(-60, 59)
        amax = rn32(F(rng.uniform(0.5, 1.0)) * F(2) ** e)
        b = rn32(amax / 448)
        mode = rng.random()
        if mode < 0.1:
            a = amax * rng.choice([1, -1])
        elif mode < 0.4:
            # quotients within a few fp32 ulps of an e4m3 rounding midpoint
            mid = F(2 * rng.randint(8, 15) + 1, 32) * F(2) ** rng.randint(-9, 7)
            a = rn32(mid * b * (1 + F(rng.randint(-4, 4), 2 ** 24)))
            a = a if rng.random() < 0.5 else -a
        else:
            a = rn32(amax * F(rng.uniform(-1, 1)) * F(2) ** -rng.randint(0, 14))
        yield a, b


def test_markstein_quotient_is_correctly_rounded():
    checked = 0
    for a, b in _cases(4000, 11):
        if b < F(2) ** -60 or b > F(2) ** 60:
            continue
        y = rn32(1 / b)
        want = rn32(a / b)
        if abs(want) <= F(1, 1024):
            continue
        assert markstein(a, b, y) == want, (float(a), float(b))
        checked += 1
    assert checked > 3000


def test_one_rounding_step_is_not_enough():
    """The first product alone can miss by more than half an ulp, which is
    why the kernel refines twice."""
    misses = 0
    for a, b in _cases(4000, 12):
        y = rn32(1 / b)
        misses += rn32(a * y) != rn32(a / b)
    assert misses > 0
