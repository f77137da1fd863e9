"""Exact-arithmetic helpers for the tests: fp32 round-to-nearest-even from exact rationals.

Independent of the oracle and of the CUDA path: values are Python Fractions, and every
operation is rounded to binary32 by the textbook rule (nearest, ties to even, gradual
underflow below 2^-126, overflow to infinity at 2^128 after rounding).
"""
from fractions import Fraction

import numpy as np

EMIN = -126          # smallest normal exponent of binary32
PREC = 24            # significand bits, hidden bit included
EMAX_BOUND = Fraction(2) ** 128


def F(x) -> Fraction:
    """Exact rational value of a finite fp32 (or any float)."""
    return Fraction(float(np.float32(x)))


def f32(q: Fraction) -> np.float32:
    """Round an exact rational to binary32, nearest-even, with subnormals."""
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    # now 2^e <= a < 2^(e+1)
    quantum_exp = max(e, EMIN) - (PREC - 1)
    scaled = a / (Fraction(2) ** quantum_exp)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = Fraction(n) * Fraction(2) ** quantum_exp
    if val >= EMAX_BOUND:
        return np.float32(sign * np.inf)
    return np.float32(sign * float(val))


def add(a, b):
    return f32(F(a) + F(b))


def mul(a, b):
    return f32(F(a) * F(b))


def div(a, b):
    return f32(F(a) / F(b))


def bits(x) -> int:
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0])


def parse_exact(tok: str) -> Fraction:
    """'1', '0', '2^-24', '1+2^-23', '2^-12', '11184813*2^-25' -> Fraction."""
    tot = Fraction(0)
    for part in tok.split("+"):
        part = part.strip()
        coef = Fraction(1)
        if "*" in part:
            c, part = part.split("*")
            coef = Fraction(int(c))
        if "^" in part:
            base, ex = part.split("^")
            tot += coef * Fraction(int(base)) ** int(ex)
        else:
            tot += coef * Fraction(part)
    return tot


def eval_shape(expr: str, leaves, combine):
    """Evaluate a fully parenthesised expression like '((0+1)+2)' over leaves by index."""
    pos = 0

    def parse():
        nonlocal pos
        if expr[pos] == "(":
            pos += 1
            left = parse()
            assert expr[pos] == "+", expr[pos:]
            pos += 1
            right = parse()
            assert expr[pos] == ")", expr[pos:]
            pos += 1
            return combine(left, right)
        start = pos
        while pos < len(expr) and expr[pos].isdigit():
            pos += 1
        return leaves[int(expr[start:pos])]

    out = parse()
    assert pos == len(expr)
    return out


def load_shapes(path):
    shapes = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, e = line.split(":", 1)
        shapes[int(k)] = e.strip()
    return shapes
