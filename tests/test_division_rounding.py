"""The quantisers on the GPU form x / scale without a division instruction:
y = RN(x r) with r = RN(1 / scale), then two correction steps
q = RN(q + RN(x - scale q) r) (one fused multiply-add each).  This checks, in
exact rational arithmetic, that the result is the correctly rounded float32
quotient -- the IEEE division the oracle uses -- for the operand ranges the
quantisers see (scale >= 2^-100, |x| <= 448 scale), on random and on
adversarial operands (quotients at and next to E4M3 tie points, scales with
all-ones and power-of-two significands)."""
from fractions import Fraction

import numpy as np


def rn32(v: Fraction) -> Fraction:
    """Round a rational to the nearest float32 (ties to even), exactly."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                                    # subnormal range: fixed quantum
    quantum = Fraction(2) ** (e - 23)
    m = a / quantum
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * quantum


def F(v) -> Fraction:
    return v if isinstance(v, Fraction) else Fraction(float(v))


def f32(v: Fraction) -> np.float32:
    return np.float32(float(v))                         # exact: v is a float32 value


def fma(a, b, c) -> Fraction:
    return rn32(F(a) * F(b) + F(c))


def quotient(x: np.float32, s: np.float32) -> np.float32:
    r = rn32(1 / F(s))
    y = rn32(F(x) * r)
    q1 = fma(fma(-F(s), y, x), r, y)
    q2 = fma(fma(-F(s), q1, x), r, q1)
    v = f32(abs(q2))
    return -v if np.signbit(x) else v                  # the sign is taken from x


def check(xs, ss):
    bad = []
    for x, s in zip(xs, ss):
        x, s = np.float32(x), np.float32(s)
        want = f32(abs(rn32(F(x) / F(s))))
        want = -want if np.signbit(x) else want          # IEEE: x / s keeps x's sign (s > 0)
        got = quotient(x, s)
        if got != want or np.signbit(got) != np.signbit(want):
            bad.append((float(x), float(s), float(got), float(want)))
    assert not bad, bad[:5]


def test_random_operands():
    rng = np.random.default_rng(3)
    n = 4000
    s = (rng.uniform(1.0, 2.0, n) * 2.0 ** rng.integers(-100, 100, n)).astype(np.float32)
    q = (rng.uniform(-448.0, 448.0, n) * 2.0 ** -rng.integers(0, 14, n)).astype(np.float32)
    x = (q.astype(np.float64) * s.astype(np.float64)).astype(np.float32)
    check(x, s)


def test_quotients_at_and_next_to_tie_points():
    rng = np.random.default_rng(4)
    xs, ss = [], []
    for _ in range(1500):
        s = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** rng.integers(-60, 60))
        e = int(rng.integers(-6, 9))
        t = (1 + (2 * int(rng.integers(0, 8)) + 1) / 16) * 2.0 ** e   # an E4M3 tie point
        x0 = np.float32(t * float(s))
        for k in (-2, -1, 0, 1, 2):                                   # neighbouring x
            xs.append(np.nextafter(x0, np.float32(np.inf) if k > 0 else np.float32(-np.inf))
                      if k else x0)
            if abs(k) == 2:
                xs[-1] = np.nextafter(xs[-1], np.float32(np.inf) if k > 0 else np.float32(-np.inf))
            ss.append(s)
    check(xs, ss)


def test_special_significands_and_signs():
    rng = np.random.default_rng(5)
    xs, ss = [], []
    for e in range(-40, 40, 3):
        for sig in (1.0, np.float32(2.0) - np.float32(2.0 ** -23), 1.5):
            s = np.float32(sig * 2.0 ** e)
            for x in rng.uniform(-448, 448, 20):
                xs.append(np.float32(x * float(s)))
                ss.append(s)
            xs += [np.float32(0.0), np.float32(-0.0), np.float32(448.0) * s, -np.float32(448.0) * s]
            ss += [s] * 4
    check(xs, ss)
