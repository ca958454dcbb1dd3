"""Exact rational Newton-Schulz on tiny matrices (pure Python integers).

TEST INFRASTRUCTURE, like ``oracle/ns64.py``: only tests and the CPU baseline may use it.

It runs the same two algorithms as ``ns64`` -- direct NS ("Newton-Schulz 变体", section
"直接空间 NS（经典）") and Gram NS with restarts (sections "Gram 空间 NS（Dao-AILab）" and
"重启机制") -- but without rounding. A value is a pair (N, D): an integer matrix N (list of rows)
and one positive integer denominator D, meaning N / D. Inputs are binary floats (exact dyadic
rationals) and the printed decimal coefficients (exact decimal rationals), so every intermediate
is an exact rational and no gcd reduction is needed to stay exact.

In exact arithmetic the Gram recurrence reproduces the direct iteration for every restart list:
X_{k+1} = (a I + Z_k) X_k, so Q_{k+1} X_0 = X_{k+1} and R_{k+1} = X_{k+1} X_{k+1}^T. Equality of the
two results is therefore a check on the Gram algorithm that owes nothing to rounding.
"""

from __future__ import annotations

from fractions import Fraction


def _lcm(a, b):
    from math import gcd
    return a // gcd(a, b) * b


def from_floats(rows):
    """Exact (N, D) for a matrix of Python floats (each float is a dyadic rational)."""
    fr = [[Fraction(float(v)) for v in row] for row in rows]
    den = 1
    for row in fr:
        for v in row:
            den = _lcm(den, v.denominator)
    return [[int(v * den) for v in row] for row in fr], den


def scalar(value):
    """Exact (p, q) of a printed decimal coefficient, read from its shortest repr."""
    f = Fraction(repr(float(value))) if not isinstance(value, (str, Fraction)) else Fraction(value)
    return f.numerator, f.denominator


def identity(n):
    return [[1 if i == j else 0 for j in range(n)] for i in range(n)], 1


def transpose(a):
    n, d = a
    return [list(col) for col in zip(*n)], d


def matmul(a, b):
    na, da = a
    nb, db = b
    cols = list(zip(*nb))
    return [[sum(x * y for x, y in zip(row, col)) for col in cols] for row in na], da * db


def scale(s, a):
    """(p/q) * A."""
    p, q = s
    n, d = a
    return [[p * v for v in row] for row in n], q * d


def add(a, b):
    na, da = a
    nb, db = b
    l = _lcm(da, db)
    fa, fb = l // da, l // db
    return [[x * fa + y * fb for x, y in zip(ra, rb)] for ra, rb in zip(na, nb)], l


def to_fractions(a):
    n, d = a
    return [[Fraction(v, d) for v in row] for row in n]


def to_floats(a):
    return [[float(v) for v in row] for row in to_fractions(a)]


def equal(a, b):
    """Exact equality of two rational matrices."""
    na, da = a
    nb, db = b
    return all(x * db == y * da for ra, rb in zip(na, nb) for x, y in zip(ra, rb))


def ns_direct(x, coeffs):
    """X <- a X + b (X X^T) X + c (X X^T)^2 X, exactly."""
    for a, b, c in coeffs:
        gram = matmul(x, transpose(x))
        gx = matmul(gram, x)
        ggx = matmul(matmul(gram, gram), x)
        x = add(add(scale(scalar(a), x), scale(scalar(b), gx)), scale(scalar(c), ggx))
    return x


def ns_gram(x, coeffs, restarts=(2,)):
    """Gram NS with restarts, exactly: same step order as the float64 oracle."""
    m = len(x[0])
    eye = identity(m)
    r = matmul(x, transpose(x))
    q = eye
    rs = set(int(k) for k in restarts)
    for k, (a, b, c) in enumerate(coeffs):
        if k in rs and k > 0:
            x = matmul(q, x)
            r = matmul(x, transpose(x))
            q = eye
        sa, sb, sc = scalar(a), scalar(b), scalar(c)
        z = add(scale(sb, r), scale(sc, matmul(r, r)))
        q = add(matmul(z, q), scale(sa, q))
        w = add(scale(sa, eye), z)
        r = matmul(matmul(w, r), w)
    return matmul(q, x)
