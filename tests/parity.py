"""Comparison rule for the CUDA path against the oracle.

Pass iff, for every checked element,
    |gpu - oracle| <= 2 * ulp16(oracle) + 1e-3 * sqrt(K),
where oracle is the exact product rounded once to fp16 and ulp16 is the fp16
spacing at that value; no NaN or Inf may appear in the GPU output.  On inputs
in {-1, 0, 1} with K <= 2048 every partial sum is an integer of magnitude at
most 2048, exact in fp32 in any order, so there the outputs must be equal
(compared by value: +0 == -0).  With ReLU no output may carry a sign bit.
"""

from __future__ import annotations

import numpy as np

import oracle


def tolerance(ref16, K: int) -> np.ndarray:
    return 2.0 * oracle.ulp16(np.asarray(ref16, dtype=np.float64)) + 1e-3 * np.sqrt(max(K, 0))


def check(gpu16, ref16, K: int, *, exact: bool = False, relu: bool = False, what: str = ""):
    g = np.asarray(gpu16, dtype=np.float16).astype(np.float64)
    r = np.asarray(ref16, dtype=np.float16).astype(np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    if relu:
        assert not np.any(np.signbit(g)), f"{what}: negative or -0 output with ReLU"
    if exact:
        bad = g != r
        assert not np.any(bad), (f"{what}: {int(bad.sum())} of {g.size} differ; first at "
                                 f"{np.argwhere(bad)[:5].tolist()}")
        return
    err = np.abs(g - r)
    tol = tolerance(r, K)
    bad = err > tol
    assert not np.any(bad), (
        f"{what}: {int(bad.sum())} of {g.size} outside tolerance; worst err "
        f"{err.max():.4g} at {np.unravel_index(np.argmax(err - tol), err.shape)}")
