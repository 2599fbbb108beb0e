"""Exact rational arithmetic used to pin the oracle (independent of its C code).

``rne_f16`` / ``rne_bf16`` round an exact rational to the nearest binary16 /
bfloat16 value, ties to even, straight from the definitions of the formats
(binary16: 11 significant bits, smallest normal 2^-14, largest 65504;
bfloat16: 8 significant bits, smallest normal 2^-126, largest
(2 - 2^-7)·2^127).  Decoding of inputs goes through numpy's float16 and
float32 types, independent implementations.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

HALF = Fraction(1, 2)


def frac_of_f16(x) -> Fraction:
    return Fraction(float(np.float16(x)))


def rne_binary(q: Fraction, mant_bits: int, emin: int, max_finite: Fraction) -> float:
    """Round the rational q to the nearest value of a binary format with
    ``mant_bits`` significant bits (hidden bit included) and smallest normal
    exponent ``emin``, ties to even; beyond ``max_finite`` (after rounding) the
    result is ±inf.  Returns the value as a float."""
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
    quantum = two ** (max(e, emin) - (mant_bits - 1))
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > HALF or (rem == HALF and fl % 2 == 1):
        fl += 1
    v = fl * quantum
    if v > max_finite:
        return s * math.inf
    return s * float(v)


def rne_f16(q: Fraction) -> float:
    """binary16: 11 significant bits, smallest normal 2^-14, largest 65504."""
    return rne_binary(q, 11, -14, Fraction(65504))


BF16_MAX = (Fraction(2) - Fraction(1, 2 ** 7)) * Fraction(2) ** 127


def rne_bf16(q: Fraction) -> float:
    """bfloat16: 8 significant bits, smallest normal 2^-126, largest (2-2^-7)·2^127."""
    return rne_binary(q, 8, -126, BF16_MAX)


F32_MAX = (Fraction(2) - Fraction(1, 2 ** 23)) * Fraction(2) ** 127


def rne_f32(q: Fraction) -> float:
    """binary32: 24 significant bits, smallest normal 2^-126, largest (2-2^-23)·2^127."""
    return rne_binary(q, 24, -126, F32_MAX)


def bf16_bits_to_float(bits) -> np.ndarray:
    """Decode bfloat16 bit patterns through numpy's binary32 (bf16 is its top half)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
        return b.view(np.float32).astype(np.float64)


def exact_gemm(A16: np.ndarray, B16: np.ndarray, relu: bool, dtype: str = "f16"):
    """Exact rational C = epi(A·B) for tiny matrices (M×K, K×N), float16 or,
    with dtype "bf16", bfloat16 bit patterns.  Returns (C rounded to the storage
    format as a float64 array, exact Fractions nested list)."""
    M, K = A16.shape
    K2, N = B16.shape
    assert K == K2
    if dtype == "bf16":
        Ad, Bd, rne = bf16_bits_to_float(A16), bf16_bits_to_float(B16), rne_bf16
    else:
        Ad, Bd, rne = A16.astype(np.float64), B16.astype(np.float64), rne_f16
    Af = [[Fraction(float(Ad[i, k])) for k in range(K)] for i in range(M)]
    Bf = [[Fraction(float(Bd[k, j])) for j in range(N)] for k in range(K)]
    out = np.empty((M, N), dtype=np.float64)
    ex = []
    for i in range(M):
        row = []
        for j in range(N):
            s = sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0))
            if relu and s < 0:
                s = Fraction(0)
            row.append(s)
            out[i, j] = rne(s)
        ex.append(row)
    return out, ex
