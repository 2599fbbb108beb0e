"""Comparison rule for the CUDA path against the oracle.

Pass iff, for every checked element,
    |gpu - oracle| <= 2 * ulp16(oracle) + 1e-3 * sqrt(K),
where oracle is the exact product rounded once to fp16 and ulp16 is the fp16
spacing at that value; no NaN or Inf may appear in the GPU output.  On inputs
in {-1, 0, 1} with K <= 2048 every partial sum is an integer of magnitude at
most 2048, exact in fp32 in any order, so there the outputs must be equal
(compared by value: +0 == -0).  With ReLU no output may carry a sign bit.
The bfloat16 variant uses the same rule with bfloat16's spacing (ulp_bf16):
its output rounding is once, like fp16's, and the 1e-3·sqrt(K) term covers
the fp32 accumulation order, which does not depend on the storage format.
"""

from __future__ import annotations

import numpy as np

import oracle


def tolerance(ref16, K: int, fmt: str = "f16") -> np.ndarray:
    ulp = oracle.ulp_bf16 if fmt == "bf16" else oracle.ulp16
    return 2.0 * ulp(np.asarray(ref16, dtype=np.float64)) + 1e-3 * np.sqrt(max(K, 0))


def check(gpu16, ref16, K: int, *, exact: bool = False, relu: bool = False, what: str = "",
          fmt: str = "f16"):
    """fmt "f16": arrays of float16 values.  fmt "bf16": arrays of float64
    values that are bfloat16 numbers (decoded from their bits)."""
    if fmt == "bf16":
        g = np.asarray(gpu16, dtype=np.float64)
        r = np.asarray(ref16, dtype=np.float64)
    else:
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
    tol = tolerance(r, K, fmt)
    bad = err > tol
    assert not np.any(bad), (
        f"{what}: {int(bad.sum())} of {g.size} outside tolerance; worst err "
        f"{err.max():.4g} at {np.unravel_index(np.argmax(err - tol), err.shape)}")
