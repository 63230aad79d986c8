"""Exact rational arithmetic used to pin the oracle (independent of it).

Every finite float32 is m * 2**e with integer m; a dot product of float32
vectors is therefore an exact rational, which Python integers hold without
rounding.  ``round_f32`` rounds such a rational to the nearest float32, ties
to even, by comparing exact distances to the neighbouring floats.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

_SHIFT = 400  # frexp exponents of float32 are >= -172 (m scaled to 24 bits), so u+v+_SHIFT >= 56


def _int_scaled(x: np.ndarray):
    """float32 array -> (integer mantissas, exponents) with x = m * 2**e exactly."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    mant, exp = np.frexp(x)                      # x = mant * 2**exp, 0.5 <= |mant| < 1
    m = np.rint(mant * (1 << 24)).astype(np.int64)
    e = exp.astype(np.int64) - 24
    return m, e


def exact_dot(a: np.ndarray, b: np.ndarray) -> Fraction:
    """sum_k a[k] * b[k] exactly."""
    ma, ea = _int_scaled(a)
    mb, eb = _int_scaled(b)
    total = 0
    for x, y, u, v in zip(ma.tolist(), mb.tolist(), ea.tolist(), eb.tolist()):
        if x and y:
            total += (x * y) << (u + v + _SHIFT)
    return Fraction(total, 1 << _SHIFT)


def exact_abs_dot(a: np.ndarray, b: np.ndarray) -> Fraction:
    return exact_dot(np.abs(a), np.abs(b))


def round_f32(q: Fraction) -> np.float32:
    """Nearest float32 to the rational q, ties to even (finite range only)."""
    guess = np.float32(float(q))
    cands = {guess, np.nextafter(guess, np.float32(-np.inf)), np.nextafter(guess, np.float32(np.inf))}
    best = None
    for c in cands:
        d = abs(q - Fraction(float(c)))
        key = (d, int(np.float32(c).view(np.uint32)) & 1)   # prefer even mantissa on a tie
        if best is None or key < best[0]:
            best = (key, c)
    out = np.float32(best[1])
    return np.float32(0.0) if out == 0 else out            # canonical +0


def exact_product(A: np.ndarray, B: np.ndarray):
    """Exact C (list of Fractions) for small A @ B."""
    M, K = A.shape
    N = B.shape[1]
    return [[exact_dot(A[i, :], B[:, j]) for j in range(N)] for i in range(M)]


def ulp_f32(x) -> float:
    x = np.float32(abs(x))
    return float(np.nextafter(x, np.float32(np.inf)) - x)
