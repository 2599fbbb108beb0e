"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with:
  * IEEE binary16 itself (numpy's float16 decoder, exact midpoints, the
    overflow threshold 65520, subnormal spacing 2^-24);
  * exact rational arithmetic (``exact.py``) on tiny products;
  * closed forms: identity and permutation B, rank-1 A, A·1 row sums;
  * integer products in {-1,0,1} against numpy's int64 matmul;
  * torch's fp64 CPU matmul (a library routine);
  * the ReLU rule (epi applied to the un-rounded sum; -0 becomes +0);
  * the leading-dimension contract (padding is never read).

The same pins run against deliberately broken builds of the oracle source in
``test_oracle_mutants.py``; every plausible mistake listed there must trip at
least one of them.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

from exact import (BF16_MAX, bf16_bits_to_float, exact_gemm, frac_of_f16, rne_bf16, rne_f16,
                   rne_f32)

ALL16 = np.arange(65536, dtype=np.uint16)


def _f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def _same_value(a, b):
    """Equal by value (+0 == -0), NaN equal to NaN."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.all((a == b) | (np.isnan(a) & np.isnan(b)))


# ---------------------------------------------------------------- binary16

def pin_decode_matches_numpy(o):
    mine = o.f64_from_f16(ALL16)
    ref = ALL16.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # sign of zero too
    assert np.signbit(mine[0x8000]) and not np.signbit(mine[0])


def pin_roundtrip_all_halves(o):
    vals = ALL16.view(np.float16).astype(np.float64)
    keep = ~np.isnan(vals)
    back = o.f16_from_f64(vals[keep])
    assert np.array_equal(back, ALL16[keep])


def pin_midpoints_tie_to_even(o):
    pos = np.arange(0, 0x7bff, dtype=np.uint16)  # pairs (h, h+1), both finite, >= 0
    lo = pos.view(np.float16).astype(np.float64)
    hi = (pos + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2.0  # exact in fp64
    got = o.f16_from_f64(mid)
    even = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint16)
    assert np.array_equal(got, even)
    # a hair either side of the midpoint goes to the nearer neighbour
    up = o.f16_from_f64(np.nextafter(mid, np.inf))
    dn = o.f16_from_f64(np.nextafter(mid, -np.inf))
    assert np.array_equal(up, pos + 1)
    assert np.array_equal(dn, pos)
    # negative side mirrors the positive side
    gotn = o.f16_from_f64(-mid)
    assert np.array_equal(gotn, even | 0x8000)


def pin_overflow_and_specials(o):
    cases = [
        (65504.0, 0x7BFF), (65519.99, 0x7BFF), (65520.0, 0x7C00), (1e6, 0x7C00),
        (-65520.0, 0xFC00), (math.inf, 0x7C00), (-math.inf, 0xFC00),
        (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000), (1.5 * 2.0 ** -25, 0x0001),
        (3 * 2.0 ** -25, 0x0002), (2.0 ** -14, 0x0400), (1.0, 0x3C00), (-2.0, 0xC000),
        (0.0, 0x0000), (-0.0, 0x8000), (1.0 + 2.0 ** -11, 0x3C00),
        (1.0 + 3 * 2.0 ** -11, 0x3C02),
    ]
    xs = np.array([c[0] for c in cases], dtype=np.float64)
    want = np.array([c[1] for c in cases], dtype=np.uint16)
    got = o.f16_from_f64(xs)
    assert np.array_equal(got, want), [(x, hex(g), hex(w)) for x, g, w in zip(xs, got, want)
                                       if g != w]
    nanbits = o.f16_from_f64(np.array([np.nan]))
    assert (nanbits[0] & 0x7C00) == 0x7C00 and (nanbits[0] & 0x3FF) != 0


def pin_matches_numpy_cast(o):
    rng = np.random.default_rng(123)
    mant = rng.uniform(1.0, 2.0, 200_000)
    expo = rng.integers(-30, 18, 200_000)
    sign = np.where(rng.integers(0, 2, 200_000) == 1, -1.0, 1.0)
    x = sign * np.ldexp(mant, expo)
    got = o.f16_from_f64(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- the product

def pin_bruteforce_exact(o):
    rng = np.random.default_rng(7)
    shapes = [(1, 1, 1), (3, 5, 7), (7, 3, 16), (16, 16, 16), (5, 9, 13), (2, 11, 4)]
    scales = [1.0, 1e-3, 64.0]  # 1e-3 puts products in the subnormal range
    for (M, N, K) in shapes:
        for sc in scales:
            A = _f16(rng.normal(0, sc, (M, K)))
            B = _f16(rng.normal(0, sc, (K, N)))
            for relu in (False, True):
                want, _ = exact_gemm(A, B, relu)
                got = o.gemm(A, B, M, N, K, relu).astype(np.float64)
                assert _same_value(got, want), (M, N, K, sc, relu, got, want)


def pin_near_tie_rounding(o):
    """Exact sums a hair off an fp16 midpoint must round from the exact value
    (a single rounding): 1 + 2^-11 is the midpoint of 1 and 1 + 2^-10."""
    t = 2.0 ** -15  # an fp16 subnormal; t*t = 2^-30
    A = _f16([[1.0, 2.0 ** -11, t], [1.0, 2.0 ** -11, -t], [1.0, 3 * 2.0 ** -11, 0.0],
              [1.0, 2.0 ** -11, 0.0]])
    B = _f16([[1.0], [1.0], [t]])
    got = o.gemm(A, B, 4, 1, 3).astype(np.float64)[:, 0]
    want = np.array([1.0 + 2.0 ** -10, 1.0, 1.0 + 2.0 ** -9, 1.0])
    assert np.array_equal(got, want), got


def pin_identity_and_permutation(o):
    rng = np.random.default_rng(11)
    M, K = 37, 29
    A = _f16(rng.uniform(-3, 3, (M, K)))
    I = np.eye(K, dtype=np.float16)
    C = o.gemm(A, I, M, K, K)
    assert np.array_equal(C.view(np.uint16) & 0x7FFF, A.view(np.uint16) & 0x7FFF)
    assert _same_value(C, A)
    Cr = o.gemm(A, I, M, K, K, relu=True)
    assert _same_value(Cr, np.maximum(A.astype(np.float64), 0.0))
    p = rng.permutation(K)
    P = np.zeros((K, K), dtype=np.float16)
    P[p, np.arange(K)] = 1.0  # B[k, j] = 1 iff k == p[j]
    Cp = o.gemm(A, P, M, K, K)
    assert _same_value(Cp, A[:, p])


def pin_rank1_and_row_sums(o):
    rng = np.random.default_rng(12)
    M, N, K = 19, 23, 41
    u = _f16(rng.uniform(-2, 2, M))
    A = np.repeat(u[:, None], K, axis=1)
    Bi = rng.integers(-4, 5, (K, N))
    B = Bi.astype(np.float16)
    C = o.gemm(A, B, M, N, K).astype(np.float64)
    colsum = Bi.sum(axis=0)
    want = np.array([[rne_f16(frac_of_f16(u[i]) * int(colsum[j])) for j in range(N)]
                     for i in range(M)])
    assert _same_value(C, want)
    # A·1: every column equals the (rounded) row sum of A
    A2 = _f16(rng.uniform(-1, 1, (M, K)))
    ones = np.ones((K, 5), dtype=np.float16)
    C2 = o.gemm(A2, ones, M, 5, K).astype(np.float64)
    rs = [rne_f16(sum((frac_of_f16(x) for x in A2[i]), Fraction(0))) for i in range(M)]
    assert _same_value(C2, np.repeat(np.array(rs)[:, None], 5, axis=1))


def pin_integer_product(o):
    rng = np.random.default_rng(13)
    M, N, K = 48, 40, 200
    Ai = rng.integers(-1, 2, (M, K))
    Bi = rng.integers(-1, 2, (K, N))
    C = o.gemm(Ai.astype(np.float16), Bi.astype(np.float16), M, N, K).astype(np.float64)
    assert np.array_equal(C, (Ai @ Bi).astype(np.float64))
    Cr = o.gemm(Ai.astype(np.float16), Bi.astype(np.float16), M, N, K, relu=True)
    assert np.array_equal(Cr.astype(np.float64), np.maximum(Ai @ Bi, 0).astype(np.float64))


def pin_torch_fp64(o):
    import torch
    rng = np.random.default_rng(14)
    M, N, K = 33, 45, 300
    A = _f16(rng.uniform(-1, 1, (M, K)))
    B = _f16(rng.uniform(-1, 1, (K, N)))
    C, ref = o.gemm(A, B, M, N, K, want_ref=True)
    t = (torch.from_numpy(A.astype(np.float64)) @ torch.from_numpy(B.astype(np.float64))).numpy()
    assert np.max(np.abs(ref - t)) <= 1e-12 * K
    assert np.mean(C.astype(np.float64) == t.astype(np.float16).astype(np.float64)) > 0.999


def pin_relu_rule(o):
    rng = np.random.default_rng(15)
    M, N, K = 31, 27, 64
    A = _f16(rng.uniform(-1, 1, (M, K)))
    B = _f16(rng.uniform(-1, 1, (K, N)))
    C0 = o.gemm(A, B, M, N, K).astype(np.float64)
    C1 = o.gemm(A, B, M, N, K, relu=True)
    assert not np.any(np.signbit(C1.astype(np.float64)))  # no negatives, no -0
    assert _same_value(C1, np.maximum(C0, 0.0))
    assert np.any(C0 < 0) and np.any(C0 > 0)
    # all-zero rows: sum is exactly 0 -> +0 with ReLU
    Z = np.zeros((2, K), dtype=np.float16)
    Z[1] = -0.0
    Cz = o.gemm(Z, B, 2, N, K, relu=True)
    assert not np.any(np.signbit(Cz.astype(np.float64)))


def pin_leading_dims(o):
    rng = np.random.default_rng(16)
    M, N, K = 9, 13, 21
    A = _f16(rng.uniform(-1, 1, (M, K)))
    B = _f16(rng.uniform(-1, 1, (K, N)))
    base = o.gemm(A, B, M, N, K)
    Ap = np.full((M, K + 11), np.nan, dtype=np.float16)
    Ap[:, :K] = A
    Bp = np.full((K, N + 3), np.inf, dtype=np.float16)
    Bp[:, :N] = B
    padded = o.gemm(Ap, Bp, M, N, K)
    assert np.array_equal(base.view(np.uint16), padded.view(np.uint16))
    want, _ = exact_gemm(A, B, False)
    assert _same_value(base, want)


def pin_sampled_matches_full(o):
    rng = np.random.default_rng(17)
    M, N, K = 70, 90, 130
    A = _f16(rng.normal(0, 1, (M, K)))
    B = _f16(rng.normal(0, 1, (K, N)))
    for relu in (False, True):
        C, ref = o.gemm(A, B, M, N, K, relu=relu, want_ref=True)
        r = rng.integers(0, M, 500)
        c = rng.integers(0, N, 500)
        v16, v64 = o.gemm_at(A, B, K, r, c, relu=relu)
        assert np.array_equal(v16.view(np.uint16), C.view(np.uint16)[r, c])
        assert np.array_equal(v64, ref[r, c])
        # and the sampled value itself is the exact sum rounded once
        for t in range(8):
            i, j = int(r[t]), int(c[t])
            s = sum((frac_of_f16(A[i, k]) * frac_of_f16(B[k, j]) for k in range(K)), Fraction(0))
            if relu and s < 0:
                s = Fraction(0)
            assert float(v16[t]) == rne_f16(s)


def pin_zero_sizes(o):
    A = np.zeros((3, 0), dtype=np.float16)
    B = np.zeros((0, 4), dtype=np.float16)
    C = o.gemm(A, B, 3, 4, 0)
    assert C.shape == (3, 4) and np.all(C.astype(np.float64) == 0.0)
    Cr = o.gemm(A, B, 3, 4, 0, relu=True)
    assert not np.any(np.signbit(Cr.astype(np.float64)))


# ---------------------------------------------------------------- bfloat16 variant

def _bf16_bits(x):
    """Round float64 values to bfloat16 bits exactly (single rounding), via
    exact rationals — independent of the oracle."""
    return np.array([_float_to_bf16_bits(rne_bf16(Fraction(float(v)))) for v in np.ravel(x)],
                    dtype=np.uint16).reshape(np.shape(x))


def _float_to_bf16_bits(v: float) -> int:
    f32 = np.array([v], dtype=np.float32)  # exact: v is a bf16 value
    return int(f32.view(np.uint32)[0] >> 16)


def pin_bf16_decode_matches_binary32(o):
    mine = o.f64_from_bf16(ALL16)
    ref = bf16_bits_to_float(ALL16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.signbit(mine[0x8000]) and not np.signbit(mine[0])


def pin_bf16_roundtrip_and_midpoints(o):
    vals = bf16_bits_to_float(ALL16)
    keep = ~np.isnan(vals)
    assert np.array_equal(o.bf16_from_f64(vals[keep]), ALL16[keep])
    pos = np.arange(0, 0x7f7f, dtype=np.uint16)  # adjacent finite pairs (h, h+1)
    lo = bf16_bits_to_float(pos)
    hi = bf16_bits_to_float(pos + 1)
    mid = (lo + hi) / 2.0
    even = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint16)
    assert np.array_equal(o.bf16_from_f64(mid), even)
    assert np.array_equal(o.bf16_from_f64(np.nextafter(mid, np.inf)), pos + 1)
    assert np.array_equal(o.bf16_from_f64(np.nextafter(mid, -np.inf)), pos)
    assert np.array_equal(o.bf16_from_f64(-mid), even | 0x8000)


def pin_bf16_overflow_and_specials(o):
    mx = float(BF16_MAX)
    half_ulp = 2.0 ** (127 - 8)
    cases = [(mx, 0x7F7F), (mx + half_ulp * 0.99, 0x7F7F), (mx + half_ulp, 0x7F80),
             (1.5 * 2.0 ** 128, 0x7F80), (1e300, 0x7F80),
             (-(mx + half_ulp), 0xFF80), (math.inf, 0x7F80), (2.0 ** -133, 0x0001),
             (2.0 ** -134, 0x0000), (1.5 * 2.0 ** -134, 0x0001), (2.0 ** -126, 0x0080),
             (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
             (1.0 + 2.0 ** -8, 0x3F80), (1.0 + 3 * 2.0 ** -8, 0x3F82)]
    got = o.bf16_from_f64(np.array([c[0] for c in cases]))
    want = np.array([c[1] for c in cases], dtype=np.uint16)
    assert np.array_equal(got, want), [(c[0], hex(g), hex(w)) for c, g, w in zip(cases, got, want)
                                       if g != w]


def pin_bf16_matches_exact_rounding(o):
    rng = np.random.default_rng(321)
    x = np.ldexp(rng.uniform(1.0, 2.0, 3000), rng.integers(-140, 128, 3000))
    x *= np.where(rng.integers(0, 2, 3000) == 1, -1.0, 1.0)
    assert np.array_equal(o.bf16_from_f64(x), _bf16_bits(x))


def pin_bf16_bruteforce_exact(o):
    rng = np.random.default_rng(8)
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (7, 3, 16), (5, 9, 13)]:
        for sc in (1.0, 1e-30, 1e20):
            A = _bf16_bits(rng.normal(0, sc, (M, K)))
            B = _bf16_bits(rng.normal(0, sc, (K, N)))
            for relu in (False, True):
                want, _ = exact_gemm(A, B, relu, dtype="bf16")
                got = bf16_bits_to_float(o.gemm(A, B, M, N, K, relu, dtype="bf16"))
                assert _same_value(got, want), (M, N, K, sc, relu)


def pin_bf16_integer_product(o):
    """{-1,0,1} products: the sum is an exact integer; bf16 then rounds it once
    (integers above 256 are not all representable)."""
    rng = np.random.default_rng(18)
    M, N, K = 24, 20, 1500
    Ai = rng.integers(-1, 2, (M, K))
    Ai[0] = 1  # row 0 against the all-ones columns sums to K = 1500
    Bi = np.ones((K, N), dtype=np.int64)
    Bi[:, ::2] = rng.integers(-1, 2, (K, (N + 1) // 2))
    A = _bf16_bits(Ai.astype(np.float64))
    B = _bf16_bits(Bi.astype(np.float64))
    got = bf16_bits_to_float(o.gemm(A, B, M, N, K, dtype="bf16"))
    want = np.array([[rne_bf16(Fraction(int(v))) for v in row] for row in Ai @ Bi])
    assert np.array_equal(got, want)
    assert np.any(np.abs(Ai @ Bi) > 256)  # the rounding is exercised


def pin_bf16_sampled_matches_full(o):
    rng = np.random.default_rng(19)
    M, N, K = 40, 50, 90
    A = _bf16_bits(rng.normal(0, 1, (M, K)))
    B = _bf16_bits(rng.normal(0, 1, (K, N)))
    C, ref = o.gemm(A, B, M, N, K, relu=True, want_ref=True, dtype="bf16")
    r = rng.integers(0, M, 300)
    c = rng.integers(0, N, 300)
    v16, v64 = o.gemm_at(A, B, K, r, c, relu=True, dtype="bf16")
    assert np.array_equal(v16, C[r, c]) and np.array_equal(v64, ref[r, c])


# ---------------------------------------------------------------- extended epilogue

def _exact_ex(A, B, relu, bias, R, in_dtype, out_dtype):
    """Exact rational out_round(act(A·B + bias[j]) + R[i][j]) for tiny inputs."""
    dec = bf16_bits_to_float if in_dtype == "bf16" else (lambda x: np.asarray(x).astype(np.float64))
    Ad, Bd = dec(A), dec(B)
    Rd = None if R is None else dec(R)
    rne = {"f16": rne_f16, "bf16": rne_bf16, "f32": rne_f32}[out_dtype]
    M, K = Ad.shape
    N = Bd.shape[1]
    out = np.empty((M, N))
    for i in range(M):
        for j in range(N):
            q = sum((Fraction(float(Ad[i, k])) * Fraction(float(Bd[k, j])) for k in range(K)),
                    Fraction(0))
            if bias is not None:
                q += Fraction(float(np.float32(bias[j])))
            if relu and q < 0:
                q = Fraction(0)
            if Rd is not None:
                q += Fraction(float(Rd[i, j]))
            out[i, j] = rne(q)
    return out


def _ex_values(C, out_dtype):
    if out_dtype == "bf16":
        return bf16_bits_to_float(C)
    return np.asarray(C).astype(np.float64)


def pin_ex_exact_bruteforce(o):
    rng = np.random.default_rng(41)
    for in_dtype in ("f16", "bf16"):
        conv = _f16 if in_dtype == "f16" else _bf16_bits
        for (M, N, K) in [(3, 5, 7), (4, 4, 16), (1, 6, 2)]:
            A = conv(rng.normal(0, 1, (M, K)))
            B = conv(rng.normal(0, 1, (K, N)))
            R = conv(rng.normal(0, 2, (M, N + 3)))  # ldr = N + 3
            bias = rng.normal(0, 2, N).astype(np.float32)
            for out_dtype in ("f16", "bf16", "f32"):
                for relu in (False, True):
                    for bb, rr in ((None, None), (bias, None), (None, R), (bias, R)):
                        want = _exact_ex(A, B, relu, bb, None if rr is None else rr[:, :N],
                                         in_dtype, out_dtype)
                        got = _ex_values(o.gemm_ex(A, B, M, N, K, relu=relu, bias=bb, R=rr,
                                                   in_dtype=in_dtype, out_dtype=out_dtype),
                                         out_dtype)
                        assert _same_value(got, want), (in_dtype, out_dtype, relu, bb is None,
                                                        rr is None)


def pin_ex_closed_forms(o):
    rng = np.random.default_rng(42)
    M, N = 9, 11
    bias = rng.normal(0, 3, N).astype(np.float32)
    R = _f16(rng.normal(0, 3, (M, N)))
    # K = 0: C = round(act(bias) + R)
    C0 = o.gemm_ex(np.zeros((M, 0), np.float16), np.zeros((0, N), np.float16), M, N, 0,
                   relu=True, bias=bias, R=R, out_dtype="f32")
    want0 = np.maximum(bias.astype(np.float64), 0.0)[None, :] + R.astype(np.float64)
    assert np.array_equal(C0.astype(np.float64), want0.astype(np.float32).astype(np.float64))
    # identity B: C = round(A + bias) exactly representable when all are small integers
    Ai = rng.integers(-8, 9, (M, N))
    bi = rng.integers(-8, 9, N).astype(np.float32)
    Ri = rng.integers(-8, 9, (M, N))
    C1 = o.gemm_ex(Ai.astype(np.float16), np.eye(N, dtype=np.float16), M, N, N, relu=True,
                   bias=bi, R=Ri.astype(np.float16))
    assert np.array_equal(C1.astype(np.float64), np.maximum(Ai + bi, 0) + Ri)
    # no bias, no residual, same output type: the plain product
    A = _f16(rng.normal(0, 1, (M, 20)))
    B = _f16(rng.normal(0, 1, (20, N)))
    assert np.array_equal(o.gemm_ex(A, B, M, N, 20, relu=True).view(np.uint16),
                          o.gemm(A, B, M, N, 20, relu=True).view(np.uint16))


def pin_ex_sampled_matches_full(o):
    rng = np.random.default_rng(43)
    M, N, K = 30, 40, 70
    A = _bf16_bits(rng.normal(0, 1, (M, K)))
    B = _bf16_bits(rng.normal(0, 1, (K, N)))
    R = _bf16_bits(rng.normal(0, 1, (M, N + 8)))
    bias = rng.normal(0, 1, N).astype(np.float32)
    for out_dtype in ("bf16", "f32"):
        C, ref = o.gemm_ex(A, B, M, N, K, relu=True, bias=bias, R=R, in_dtype="bf16",
                           out_dtype=out_dtype, want_ref=True)
        r = rng.integers(0, M, 200)
        c = rng.integers(0, N, 200)
        v, v64 = o.gemm_ex_at(A, B, K, r, c, relu=True, bias=bias, R=R, in_dtype="bf16",
                              out_dtype=out_dtype)
        assert np.array_equal(np.asarray(v), np.asarray(C)[r, c]) and np.array_equal(v64, ref[r, c])




# ---------------------------------------------------------------- MXFP4 weights
#
# Facts from the OCP Microscaling (MX) format specification, not from the
# oracle: the FP4 E2M1 element values for codes 0..15 (sign-magnitude, codes
# 8..15 negative, code 8 is -0) and the E8M0 scale 2^(X-127) with 0xFF = NaN.

E2M1_SPEC = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
             -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def _pack_codes(codes: np.ndarray, ld_bytes: int | None = None) -> np.ndarray:
    """K×N codes (0..15) into N rows of ceil(K/2) bytes: row n holds column n's
    codes along k, low nibble = even k."""
    K, N = codes.shape
    ld = (K + 1) // 2 if ld_bytes is None else ld_bytes
    out = np.zeros((N, ld), dtype=np.uint8)
    for k in range(K):
        out[:, k // 2] |= (codes[k, :].astype(np.uint8) << (4 * (k % 2))).astype(np.uint8)
    return out


def _exact_deq(code: int, x: int) -> Fraction:
    return Fraction(E2M1_SPEC[code]) * (Fraction(2) ** (int(x) - 127))


def pin_mx_e2m1_table(o):
    for code, want in enumerate(E2M1_SPEC):
        got = o.e2m1(code)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), (code, got)


def pin_mx_e8m0(o):
    assert o.e8m0(127) == 1.0
    assert o.e8m0(128) == 2.0 and o.e8m0(126) == 0.5
    assert o.e8m0(0) == float(Fraction(1, 2 ** 127))
    assert o.e8m0(254) == float(2 ** 127)
    assert math.isnan(o.e8m0(255))


def pin_mx_dequant_exact(o):
    """Every (code, scale) pair over a scale range that covers underflow to
    zero, fp16 subnormals, normals and overflow to inf, against exact
    rational rounding; also fixes the nibble order and the scale indexing."""
    rng = np.random.default_rng(51)
    K, N = 71, 37  # ragged: three scale rows, odd K (a padding nibble)
    codes = rng.integers(0, 16, (K, N))
    X = rng.integers(95, 146, ((K + 31) // 32, N)).astype(np.uint8)
    Bq = _pack_codes(codes, ld_bytes=40)
    got = o.mxfp4_dequant(Bq, X, K, N).astype(np.float64)
    for k in range(K):
        for n in range(N):
            want = rne_f16(_exact_deq(int(codes[k, n]), int(X[k // 32, n])))
            if want == 0.0:  # a zero result keeps the element's sign (code bit 3)
                want = math.copysign(0.0, -1.0 if codes[k, n] >= 8 else 1.0)
            g = got[k, n]
            assert (g == want and math.copysign(1, g) == math.copysign(1, want)), \
                (k, n, int(codes[k, n]), int(X[k // 32, n]), g, want)
    # NaN scale: every element of that block is NaN
    X2 = X.copy()
    X2[1, 3] = 255
    d2 = o.mxfp4_dequant(Bq, X2, K, N).astype(np.float64)
    assert np.all(np.isnan(d2[32:64, 3])) and not np.any(np.isnan(d2[:32, 3]))


def pin_mx_padding_ignored(o):
    """Bytes past ceil(K/2), the spare high nibble of an odd K, and scale
    columns past N are never read."""
    rng = np.random.default_rng(52)
    K, N = 41, 9
    codes = rng.integers(0, 16, (K, N))
    X = rng.integers(120, 130, ((K + 31) // 32, N + 4)).astype(np.uint8)
    Bq = _pack_codes(codes, ld_bytes=24)
    ref = o.mxfp4_dequant(Bq, X, K, N).view(np.uint16).copy()
    Bq2 = Bq.copy()
    Bq2[:, 21:] = 0xEE
    Bq2[:, 20] |= 0xF0  # high nibble of byte 20 is k = 41: padding for K = 41
    X2 = X.copy()
    X2[:, N:] = 255
    assert np.array_equal(o.mxfp4_dequant(Bq2, X2, K, N).view(np.uint16), ref)


def pin_mx_gemm_exact(o):
    """C = out(act(A·Bdeq + bias) + R) against exact rationals, with scales
    where every dequantised weight is an fp16 number (so no intermediate
    rounding is involved)."""
    rng = np.random.default_rng(53)
    M, N, K = 3, 5, 70
    A = _f16(rng.normal(0, 1, (M, K)))
    codes = rng.integers(0, 16, (K, N))
    X = rng.integers(115, 130, ((K + 31) // 32, N)).astype(np.uint8)
    Bq = _pack_codes(codes)
    bias = rng.normal(0, 1, N).astype(np.float32)
    R = _f16(rng.normal(0, 1, (M, N)))
    Ad = A.astype(np.float64)
    for relu in (False, True):
        for out_dtype in ("f16", "f32"):
            got = np.asarray(o.gemm_mxfp4(A, Bq, X, M, N, K, relu=relu, bias=bias, R=R,
                                          out_dtype=out_dtype), dtype=np.float64)
            rne = rne_f16 if out_dtype == "f16" else rne_f32
            for i in range(M):
                for j in range(N):
                    q = sum((Fraction(float(Ad[i, k])) * _exact_deq(int(codes[k, j]),
                                                                    int(X[k // 32, j]))
                             for k in range(K)), Fraction(0))
                    q += Fraction(float(bias[j]))
                    if relu and q < 0:
                        q = Fraction(0)
                    q += Fraction(float(R[i, j]))
                    assert got[i, j] == rne(q), (relu, out_dtype, i, j)


def pin_mx_gemm_integer_closed_form(o):
    """Codes ±1 (2, 10) with scale 2^0 make Bdeq a ±1 matrix: C equals
    numpy's int64 product of the integer A with that sign matrix."""
    rng = np.random.default_rng(54)
    M, N, K = 6, 10, 96
    Ai = rng.integers(-3, 4, (M, K))
    sign = rng.integers(0, 2, (K, N))
    codes = np.where(sign == 1, 10, 2)  # 2 -> +1.0, 10 -> -1.0
    X = np.full(((K + 31) // 32, N), 127, dtype=np.uint8)
    C = o.gemm_mxfp4(Ai.astype(np.float16), _pack_codes(codes), X, M, N, K)
    want = Ai @ np.where(sign == 1, -1, 1)
    assert np.array_equal(C.astype(np.float64), want.astype(np.float64))


# ---------------------------------------------------------------- 2:4 sparse A
#
# The format is fixed by its definition (tgemm_oracle.c): each group of four k
# keeps two values; a 4-bit field per group holds the first kept position in
# its low two bits and the second in its high two bits, eight groups per
# 32-bit word, group 0 in the lowest bits.  The helpers below restate that
# encoding independently (compression, not decompression).

SP24_PATTERNS = [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)]


def sp24_random(rng, M, K, values):
    """A dense 2:4 matrix (float64) with kept positions drawn per group, its
    compressed values (M × K/2) and metadata words (M × K/32 uint32)."""
    A = np.zeros((M, K))
    Ac = np.zeros((M, K // 2))
    E = np.zeros((M, K // 32), dtype=np.uint64)
    for i in range(M):
        for G in range(K // 4):
            p0, p1 = SP24_PATTERNS[rng.integers(0, 6)]
            v0, v1 = values(rng), values(rng)
            A[i, 4 * G + p0], A[i, 4 * G + p1] = v0, v1
            Ac[i, 2 * G], Ac[i, 2 * G + 1] = v0, v1
            E[i, G // 8] |= np.uint64((p0 | (p1 << 2)) << (4 * (G % 8)))
    return A, Ac, E.astype(np.uint32)


def pin_sp24_hand_example(o):
    """Two rows worked by hand from the format definition."""
    Ac = _f16(np.arange(1, 33).reshape(2, 16))
    E = np.array([[0xE4E4E4E4], [0x98DC4C4C]], dtype=np.uint32)
    A = o.sp24_decompress(Ac, E, 2, 32).view(np.float16).astype(np.float64)
    want = np.zeros((2, 32))
    # row 0: groups alternate positions (0,1) [nibble 4] and (2,3) [nibble E]
    for G in range(8):
        p = (0, 1) if G % 2 == 0 else (2, 3)
        want[0, 4 * G + p[0]], want[0, 4 * G + p[1]] = 2 * G + 1, 2 * G + 2
    # row 1: nibbles from group 0 up: C 4 C 4 C D 8 9
    for G, p in enumerate([(0, 3), (0, 1), (0, 3), (0, 1), (0, 3), (1, 3), (0, 2), (1, 2)]):
        want[1, 4 * G + p[0]], want[1, 4 * G + p[1]] = 17 + 2 * G, 18 + 2 * G
    assert np.array_equal(A, want)


def pin_sp24_roundtrip_and_exact_gemm(o):
    rng = np.random.default_rng(61)
    for (M, N, K) in [(3, 5, 32), (4, 3, 64), (1, 7, 96)]:
        A, Ac, E = sp24_random(rng, M, K, lambda r: float(np.float16(r.normal(0, 1))))
        Ac16 = _f16(Ac)
        assert np.array_equal(o.sp24_decompress(Ac16, E, M, K).view(np.float16).astype(np.float64),
                              A)
        B = _f16(rng.normal(0, 1, (K, N)))
        for relu in (False, True):
            got = o.gemm_sp24(Ac16, E, B, M, N, K, relu=relu).astype(np.float64)
            want, _ = exact_gemm(_f16(A), B, relu)
            assert _same_value(got, want), (M, N, K, relu)


def pin_sp24_invalid_metadata_rejected(o):
    Ac = _f16(np.ones((1, 16)))
    for nib in (0x0, 0x5, 0xA, 0xF, 0x1, 0x6, 0xB):  # first >= second
        E = np.array([[0xE4E4E4E0 | nib]], dtype=np.uint32)
        try:
            o.sp24_decompress(Ac, E, 1, 32)
        except ValueError:
            continue
        raise AssertionError(f"nibble {nib:#x} accepted")


def pin_sp24_padding_ignored(o):
    """Ac entries past K/2 and metadata words past K/32 are never read."""
    rng = np.random.default_rng(62)
    M, K = 3, 64
    A, Ac, E = sp24_random(rng, M, K, lambda r: float(r.integers(1, 9)))
    Acp = np.full((M, 40), np.float16(np.nan), dtype=np.float16)
    Acp[:, :32] = _f16(Ac)
    Ep = np.full((M, 5), 0xFFFFFFFF, dtype=np.uint32)  # invalid if read
    Ep[:, :2] = E
    assert np.array_equal(o.sp24_decompress(Acp, Ep, M, K).view(np.float16).astype(np.float64), A)


def pin_sp24_integer_closed_form(o):
    """Integer values: C equals numpy's int64 product of the dense A with B."""
    rng = np.random.default_rng(63)
    M, N, K = 8, 9, 128
    A, Ac, E = sp24_random(rng, M, K, lambda r: float(r.integers(-3, 4)))
    Bi = rng.integers(-2, 3, (K, N))
    C = o.gemm_sp24(_f16(Ac), E, Bi.astype(np.float16), M, N, K)
    assert np.array_equal(C.astype(np.float64), (A.astype(np.int64) @ Bi).astype(np.float64))


def pin_sp24_sampled_matches_full(o):
    """gemm_sp24_at (which decompresses only the rows it needs) equals the full
    gemm_sp24 bit for bit, on rows given out of order, repeated, and leaving
    rows out, with bias, residual (its own leading dimension) and both output
    types."""
    rng = np.random.default_rng(64)
    M, N, K = 9, 11, 96
    _, Ac, E = sp24_random(rng, M, K, lambda r: float(np.float16(r.normal(0, 1))))
    Ac16 = _f16(Ac)
    B = _f16(rng.normal(0, 1, (K, N)))
    R = _f16(rng.normal(0, 1, (M, N + 3)))
    bias = rng.normal(0, 1, N).astype(np.float32)
    # rows 0, 2 and 7 never appear, so the row subset is not the identity
    rows = np.array([8, 1, 8, 4, 3, 3, 6, 5, 1] + list(rng.choice([1, 3, 4, 5, 6, 8], 120)))
    cols = rng.integers(0, N, rows.size)
    for relu in (False, True):
        for out_dtype in ("f16", "f32"):
            C = o.gemm_sp24(Ac16, E, B, M, N, K, relu=relu, bias=bias, R=R, out_dtype=out_dtype)
            v, _ = o.gemm_sp24_at(Ac16, E, B, K, rows, cols, relu=relu, bias=bias, R=R,
                                  out_dtype=out_dtype)
            v, C = np.asarray(v), np.asarray(C)
            assert v.dtype == C.dtype, (out_dtype, v.dtype, C.dtype)
            assert np.array_equal(v.view(np.uint8), np.ascontiguousarray(C[rows, cols]).view(np.uint8)), \
                (relu, out_dtype)


def pin_mx_sampled_matches_full(o):
    """gemm_mxfp4_at equals the full gemm_mxfp4 bit for bit on scattered
    elements, with ReLU, bias, residual and both output types (K != N, so a
    swapped dimension cannot pass)."""
    rng = np.random.default_rng(55)
    M, N, K = 7, 13, 100
    A = _f16(rng.normal(0, 1, (M, K)))
    codes = rng.integers(0, 16, (K, N))
    X = rng.integers(118, 132, ((K + 31) // 32, N)).astype(np.uint8)
    Bq = _pack_codes(codes)
    R = _f16(rng.normal(0, 1, (M, N + 5)))
    bias = rng.normal(0, 1, N).astype(np.float32)
    rows = rng.integers(0, M, 150)
    cols = rng.integers(0, N, 150)
    for relu in (False, True):
        for out_dtype in ("f16", "f32"):
            C = o.gemm_mxfp4(A, Bq, X, M, N, K, relu=relu, bias=bias, R=R, out_dtype=out_dtype)
            v, _ = o.gemm_mxfp4_at(A, Bq, X, K, N, rows, cols, relu=relu, bias=bias, R=R,
                                   out_dtype=out_dtype)
            v, C = np.asarray(v), np.asarray(C)
            assert v.dtype == C.dtype, (out_dtype, v.dtype, C.dtype)
            assert np.array_equal(v.view(np.uint8), np.ascontiguousarray(C[rows, cols]).view(np.uint8)), \
                (relu, out_dtype)


# ---------------------------------------------------------------- tolerance spacings
#
# The parity tolerance is 2 spacings of the output format at the oracle value
# plus 1e-3*sqrt(K).  The spacing functions are pinned to the formats
# themselves: for every positive finite number x of the format below its
# largest, the spacing at x is the distance to the next number up, read from
# consecutive bit patterns (binary16 through numpy's decoder; bfloat16 as the
# upper half of a binary32 pattern).  Hand-picked values cover zero, the
# subnormal range, binade edges and the largest finite number.

def _bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def pin_spacing_f16_consecutive(o):
    import oracle
    h = np.arange(0, 0x7BFF, dtype=np.uint16)  # 0 .. next-to-largest finite
    x = h.view(np.float16).astype(np.float64)
    nxt = (h + 1).view(np.float16).astype(np.float64)
    assert np.array_equal(oracle.ulp16(x), nxt - x)
    assert np.array_equal(oracle.ulp16(-x), nxt - x)
    hand = {0.0: 2.0 ** -24, 1.0: 2.0 ** -10, 1.999: 2.0 ** -10, 2.0: 2.0 ** -9,
            65504.0: 32.0, 2.0 ** -14: 2.0 ** -24, 2.0 ** -15: 2.0 ** -24, -3.0: 2.0 ** -9}
    got = oracle.ulp16(np.array(list(hand)))
    assert list(got) == list(hand.values())


def pin_spacing_bf16_consecutive(o):
    import oracle
    h = np.arange(0, 0x7F7F, dtype=np.uint32)  # 0 .. next-to-largest finite
    x = _bf16_value(h)
    nxt = _bf16_value(h + 1)
    assert np.array_equal(oracle.ulp_bf16(x), nxt - x)
    assert np.array_equal(oracle.ulp_bf16(-x), nxt - x)
    bmax = float(_bf16_value(0x7F7F))  # largest finite bfloat16, (2 - 2^-7) * 2^127
    assert bmax == (2.0 - 2.0 ** -7) * 2.0 ** 127
    hand = {0.0: 2.0 ** -133, 1.0: 2.0 ** -7, 1.999: 2.0 ** -7, 2.0: 2.0 ** -6,
            bmax: 2.0 ** 120, 2.0 ** -126: 2.0 ** -133, 2.0 ** -127: 2.0 ** -133,
            -3.0: 2.0 ** -6}
    got = oracle.ulp_bf16(np.array(list(hand)))
    assert list(got) == list(hand.values())


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
