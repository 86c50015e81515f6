"""Exact-rational helpers for the oracle's pins (independent of oracle.c)."""
from fractions import Fraction

import numpy as np


def rn_f32(x: Fraction) -> float:
    """round a rational to the nearest float32, ties to even (normal range)"""
    if x == 0:
        return 0.0
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    q = a / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return float(np.float32(sign * float(n * ulp)))


def rn_f64(x: Fraction) -> float:
    """Python's int / int true division is correctly rounded"""
    return x.numerator / x.denominator
