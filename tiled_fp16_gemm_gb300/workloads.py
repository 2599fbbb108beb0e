"""Seeded synthetic workloads for the tiled FP16 GEMM C = epi(A·B).

This module only *draws inputs*: it holds no GEMM arithmetic, so both the CUDA
path and the CPU oracle can take their operands from it without sharing any
part of the method.  The shapes are the ones the library is measured on; the
pages that describe the method print no input data, so every distribution
below is a stated choice (uniform[-1, 1) as in a plain quickstart test, the
{-1, 0, 1} exactness variant, and normal(0, 1/sqrt(K)) weights for the
transformer-MLP and weight-streaming shapes).

Recipe (identical for every consumer):
  * A is drawn with ``numpy.random.default_rng([seed, 0])``, B with
    ``numpy.random.default_rng([seed, 1])``, in float64, row by row in C order,
    then cast to float16 with numpy's round-to-nearest-even cast.
  * A leading dimension larger than the row width pads each row with zeros
    (the padding is never read by a correct GEMM).
"""

from __future__ import annotations

import dataclasses
import numpy as np

__all__ = ["Workload", "WORKLOADS", "draw", "draw_inputs", "sample_positions"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    relu: bool
    dist_a: tuple  # ("uniform", lo, hi) | ("normal", mean, std) | ("ints", lo, hi_exclusive)
    dist_b: tuple
    seed: int
    note: str = ""

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        """A, B read once and C written once, fp16."""
        return 2 * (self.M * self.K + self.K * self.N + self.M * self.N)


def _u():
    return ("uniform", -1.0, 1.0)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("gemm_256", 256, 256, 256, False, _u(), _u(), 1,
                 "small square case; the oracle finishes in well under a second"),
        Workload("gemm_1024_relu", 1024, 1024, 1024, True, _u(), _u(), 2,
                 "square, fused ReLU"),
        Workload("gemm_1024_relu_int", 1024, 1024, 1024, True,
                 ("ints", -1, 2), ("ints", -1, 2), 22,
                 "exactness variant: entries in {-1,0,1}, every partial sum exact in fp32"),
        Workload("gemm_4096", 4096, 4096, 4096, False, _u(), _u(), 3,
                 "square, tensor-core bound"),
        Workload("mlp_8192x28672x4096_relu", 8192, 28672, 4096, True,
                 ("normal", 0.0, 1.0 / 64.0), ("normal", 0.0, 1.0 / 64.0), 4,
                 "transformer-MLP shaped, compute bound, fused ReLU"),
        Workload("skinny_64x16384x8192", 64, 16384, 8192, False,
                 ("normal", 0.0, 1.0), ("normal", 0.0, 1.0 / float(np.sqrt(8192.0))), 5,
                 "weight streaming, HBM bound (B is 256 MiB)"),
        Workload("profile_8192x8192x4096_relu", 8192, 8192, 4096, True,
                 ("normal", 0.0, 1.0 / 64.0), ("normal", 0.0, 1.0 / 64.0), 6,
                 "profiling case for the persistent kernel: the MLP shape with N cut to "
                 "8192 (256 MiB of A, B and C, twice L2)"),
    ]
}


def draw(rng: np.random.Generator, dist: tuple, rows: int, cols: int) -> np.ndarray:
    """Draw a rows×cols float64 matrix from ``dist`` (see ``Workload.dist_a``)."""
    kind = dist[0]
    if kind == "uniform":
        return rng.uniform(dist[1], dist[2], size=(rows, cols))
    if kind == "normal":
        return rng.normal(dist[1], dist[2], size=(rows, cols))
    if kind == "ints":
        return rng.integers(dist[1], dist[2], size=(rows, cols)).astype(np.float64)
    raise ValueError(f"unknown distribution {dist!r}")


def _pad(x16: np.ndarray, ld: int | None) -> np.ndarray:
    rows, cols = x16.shape
    if ld is None or ld == cols:
        return np.ascontiguousarray(x16)
    if ld < cols:
        raise ValueError("leading dimension smaller than the row width")
    out = np.zeros((rows, ld), dtype=np.float16)
    out[:, :cols] = x16
    return out


def draw_inputs(M: int, N: int, K: int, dist_a: tuple, dist_b: tuple, seed: int,
                lda: int | None = None, ldb: int | None = None):
    """Return (A, B) as float16 arrays of shape (M, lda) and (K, ldb)."""
    a = draw(np.random.default_rng([seed, 0]), dist_a, M, K).astype(np.float16)
    b = draw(np.random.default_rng([seed, 1]), dist_b, K, N).astype(np.float16)
    return _pad(a, lda), _pad(b, ldb)


def workload_inputs(w: Workload, lda: int | None = None, ldb: int | None = None):
    return draw_inputs(w.M, w.N, w.K, w.dist_a, w.dist_b, w.seed, lda, ldb)


def sample_positions(M: int, N: int, BM: int, BN: int, seed: int, n_random: int = 4096):
    """Output positions to check on shapes too large for a full oracle run.

    ``n_random`` (row, col) pairs drawn with ``default_rng(seed + 7)`` plus every
    element of the rows and columns that sit on tile edges of a BM×BN tiling
    (first/last row or column of the first, middle and last tile).
    Returns (rows, cols) as int64 arrays.
    """
    rng = np.random.default_rng(seed + 7)
    ri = rng.integers(0, M, size=n_random)
    ci = rng.integers(0, N, size=n_random)

    def edges(X, B):
        c = [0, B - 1, B, X // 2 - 1, X // 2, X - B - 1, X - B, X - 1]
        return sorted({v for v in c if 0 <= v < X})

    er, ec = edges(M, BM), edges(N, BN)
    rows = [ri]
    cols = [ci]
    for r in er:  # full rows
        rows.append(np.full(N, r, dtype=np.int64))
        cols.append(np.arange(N, dtype=np.int64))
    for c in ec:  # full columns
        rows.append(np.arange(M, dtype=np.int64))
        cols.append(np.full(M, c, dtype=np.int64))
    return (np.concatenate(rows).astype(np.int64), np.concatenate(cols).astype(np.int64))


# ------------------------------------------------------------------ MXFP4 weights

@dataclasses.dataclass(frozen=True)
class MxWorkload:
    """A fp16 (M×K) times an MXFP4 weight (K×N): packed E2M1 codes and E8M0
    scales, both drawn as plain random bytes (no encoder involved)."""
    name: str
    M: int
    N: int
    K: int
    relu: bool
    dist_a: tuple
    scale_lo: int  # E8M0 scale bytes drawn uniformly from [scale_lo, scale_hi]
    scale_hi: int
    seed: int
    note: str = ""

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        """A read once, packed codes (K/2 bytes per weight column) and scales
        (N per 32 k) read once, C written once (fp16)."""
        return (2 * self.M * self.K + self.N * ((self.K + 1) // 2)
                + ((self.K + 31) // 32) * self.N + 2 * self.M * self.N)


MX_WORKLOADS = {
    w.name: w
    for w in [
        MxWorkload("mxfp4_skinny_64x16384x8192", 64, 16384, 8192, False, ("normal", 0.0, 1.0),
                   118, 122, 7,
                   "weight streaming with MXFP4 weights: the skinny shape's B at 0.53 bytes "
                   "per weight (64 MiB of codes + 4 MiB of scales)"),
        MxWorkload("mxfp4_mlp_8192x28672x4096_relu", 8192, 28672, 4096, True,
                   ("normal", 0.0, 1.0 / 64.0), 118, 122, 8,
                   "the MLP shape with MXFP4 weights (dequantise-then-GEMM path)"),
    ]
}


def round16(x: int) -> int:
    return (x + 15) // 16 * 16


def draw_mxfp4(rng: np.random.Generator, K: int, N: int, scale_lo: int, scale_hi: int,
               ldbq: int | None = None, lds: int | None = None):
    """(Bq, S): N × ldbq random bytes (a weight column's codes along k, two
    4-bit codes per byte; every code value equally likely) and ceil(K/32) ×
    lds scale bytes uniform in [scale_lo, scale_hi].  Default row strides are
    rounded up to 16 bytes.  Padding bytes are random too (a correct GEMM
    never decodes them)."""
    ldbq = round16((K + 1) // 2) if ldbq is None else ldbq
    lds = round16(N) if lds is None else lds
    Bq = rng.integers(0, 256, size=(N, ldbq), dtype=np.uint8)
    S = rng.integers(scale_lo, scale_hi + 1, size=((K + 31) // 32, lds), dtype=np.uint8)
    return Bq, S


def mx_workload_inputs(w: MxWorkload):
    """(A float16 M×K, Bq, S) for an MXFP4 workload."""
    A = draw(np.random.default_rng([w.seed, 0]), w.dist_a, w.M, w.K).astype(np.float16)
    Bq, S = draw_mxfp4(np.random.default_rng([w.seed, 1]), w.K, w.N, w.scale_lo, w.scale_hi)
    return A, Bq, S


# ------------------------------------------------------------------ 2:4 sparse A

SP24_PATTERN_CODES = np.array([0x4, 0x8, 0xC, 0x9, 0xD, 0xE], dtype=np.uint32)
"""The six valid 4-bit group codes of the 2:4 metadata format (positions
(0,1), (0,2), (0,3), (1,2), (1,3), (2,3): first in the low two bits)."""


def draw_sp24(rng: np.random.Generator, M: int, K: int, dist: tuple, lde: int | None = None):
    """A random 2:4 sparse M×K matrix drawn directly in its stored form:
    kept values Ac (float16, M × K/2) from ``dist`` and metadata words E
    (uint32, M × lde, lde >= K/32) whose group codes are drawn uniformly from
    the six valid ones.  No dense matrix is formed."""
    Ac = draw(rng, dist, M, K // 2).astype(np.float16)
    codes = SP24_PATTERN_CODES[rng.integers(0, 6, size=(M, K // 4))]
    words = np.zeros((M, K // 32), dtype=np.uint32)
    for g in range(8):
        words |= codes[:, g::8] << np.uint32(4 * g)
    lde = K // 32 if lde is None else lde
    E = np.zeros((M, lde), dtype=np.uint32)
    E[:, :K // 32] = words
    return Ac, E


@dataclasses.dataclass(frozen=True)
class Sp24Workload:
    name: str
    M: int
    N: int
    K: int
    relu: bool
    dist_a: tuple
    dist_b: tuple
    seed: int
    note: str = ""

    @property
    def flops(self) -> int:
        """Dense-equivalent: 2·M·N·K (the skipped zeros counted as work)."""
        return 2 * self.M * self.N * self.K


SP24_WORKLOADS = {
    w.name: w
    for w in [
        Sp24Workload("sp24_mlp_8192x28672x4096_relu", 8192, 28672, 4096, True,
                     ("normal", 0.0, 1.0 / 64.0), ("normal", 0.0, 1.0 / 64.0), 9,
                     "the MLP shape with a 2:4 sparse A (half of A's weights pruned)"),
        Sp24Workload("sp24_8192x8192x4096_relu", 8192, 8192, 4096, True,
                     ("normal", 0.0, 1.0 / 64.0), ("normal", 0.0, 1.0 / 64.0), 10,
                     "a smaller square case for profiling captures: 228 MB of operands "
                     "and output, above the L2's 129 MB"),
    ]
}


def sp24_workload_inputs(w: Sp24Workload):
    """(Ac, E, B) for a 2:4 workload."""
    Ac, E = draw_sp24(np.random.default_rng([w.seed, 0]), w.M, w.K, w.dist_a)
    B = draw(np.random.default_rng([w.seed, 1]), w.dist_b, w.K, w.N).astype(np.float16)
    return Ac, E, B
