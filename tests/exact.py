"""Exact rational arithmetic used to pin the oracle (independent of its C code).

``rne_f16`` rounds an exact rational to the nearest binary16 value, ties to
even, straight from the definition of the format (1 sign bit, 5 exponent bits
with bias 15, 10 fraction bits; subnormal spacing 2^-24; largest finite value
65504).  Decoding of fp16 inputs goes through numpy's float16 type, another
independent implementation.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

HALF = Fraction(1, 2)


def frac_of_f16(x) -> Fraction:
    return Fraction(float(np.float16(x)))


def rne_f16(q: Fraction) -> float:
    """Round the rational q to binary16 (RNE); returns the value as a float."""
    if q == 0:
        return 0.0
    s = -1.0 if q < 0 else 1.0
    a = -q if q < 0 else q
    e = a.numerator.bit_length() - a.denominator.bit_length()
    two = Fraction(2)
    while two ** e > a:
        e -= 1
    while two ** (e + 1) <= a:
        e += 1
    quantum = Fraction(1, 2 ** 24) if e < -14 else two ** (e - 10)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > HALF or (rem == HALF and fl % 2 == 1):
        fl += 1
    v = fl * quantum
    if v > 65504:
        return s * math.inf
    return s * float(v)


def exact_gemm(A16: np.ndarray, B16: np.ndarray, relu: bool):
    """Exact rational C = epi(A·B) for tiny float16 matrices (M×K, K×N).
    Returns (C rounded to fp16 as float64 array, exact Fractions nested list)."""
    M, K = A16.shape
    K2, N = B16.shape
    assert K == K2
    Af = [[frac_of_f16(A16[i, k]) for k in range(K)] for i in range(M)]
    Bf = [[frac_of_f16(B16[k, j]) for j in range(N)] for k in range(K)]
    out = np.empty((M, N), dtype=np.float64)
    ex = []
    for i in range(M):
        row = []
        for j in range(N):
            s = sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0))
            if relu and s < 0:
                s = Fraction(0)
            row.append(s)
            out[i, j] = rne_f16(s)
        ex.append(row)
    return out, ex
