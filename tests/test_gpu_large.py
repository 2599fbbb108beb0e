"""Sizes at the far end: a C of more than 2^31 elements, a million rows of A,
K of a million, N of four million on the M <= 128 kernel.  Each is checked
against the oracle on sampled elements (random ones, every pair of tile-edge
row and column, the last 2048 of each edge row and column; the oracle
evaluates only those), and, where integer inputs make every partial sum exact
in fp32 (|sum| <= 2^20 < 2^24), for exact equality.  The samples are gathered
on the device, so only they travel to the host.
"""

import numpy as np
import pytest

import oracle
from parity import check

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from tiled_fp16_gemm_gb300 import workloads as W  # noqa: E402


@pytest.fixture(scope="module")
def tg():
    from tiled_fp16_gemm_gb300 import build
    build.build()
    import tiled_fp16_gemm_gb300 as t
    return t


def _edges(X, B):
    c = [0, B - 1, B, X // 2 - 1, X // 2, X - B - 1, X - B, X - 1]
    return sorted({v for v in c if 0 <= v < X})


def _positions(M, N, seed, extra_rows=()):
    """Random elements, every pair of tile-edge row and column (256 x 256
    tiles), the runs of 2048 elements that end each edge row and column, and
    64 random elements of each extra row."""
    rng = np.random.default_rng(seed)
    er, ec = _edges(M, 256), _edges(N, 256)
    rows = [rng.integers(0, M, 20000)]
    cols = [rng.integers(0, N, 20000)]
    rr, cc = np.meshgrid(np.asarray(er), np.asarray(ec), indexing="ij")
    rows.append(rr.ravel())
    cols.append(cc.ravel())
    for r in er:
        n = min(N, 2048)
        rows.append(np.full(n, r))
        cols.append(np.arange(N - n, N))
    for c in ec:
        n = min(M, 2048)
        rows.append(np.arange(M - n, M))
        cols.append(np.full(n, c))
    for r in extra_rows:
        rows.append(np.full(64, r))
        cols.append(rng.integers(0, N, 64))
    return (np.concatenate(rows).astype(np.int64), np.concatenate(cols).astype(np.int64))


def _run_sampled(tg, A, B, M, N, K, rows, cols, relu):
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    tg.gemm(a, b, relu=relu, out=c)
    tg.sync_status()
    r = torch.from_numpy(rows).cuda()
    q = torch.from_numpy(cols).cuda()
    got = c[r, q].cpu().numpy()
    del a, b, c
    torch.cuda.empty_cache()
    return got


@pytest.mark.parametrize("dist", ["normal", "ints"])
def test_c_beyond_2_pow_31_elements(tg, monkeypatch, dist):
    """65536 x 34816 = 2.28e9 elements of C (4.6 GB): element offsets past
    2^31, rows past 2^31 / N included."""
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M, N, K = 65536, 34816, 64
    assert M * N > 2 ** 31
    if dist == "ints":
        A, B = W.draw_inputs(M, N, K, ("ints", -1, 2), ("ints", -1, 2), 31)
    else:
        A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), 31)
    first_past = 2 ** 31 // N + 1
    rows, cols = _positions(M, N, 41, extra_rows=(first_past, first_past + 1, M - 2))
    got = _run_sampled(tg, A, B, M, N, K, rows, cols, relu=False)
    want, _ = oracle.gemm_at(A, B, K, rows, cols)
    check(got, want, K, exact=(dist == "ints"), what=f"{M}x{N}x{K} {dist}")


def test_a_million_rows(tg, monkeypatch):
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M, N, K = 1 << 20, 192, 96
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), 32)
    rows, cols = _positions(M, N, 42)
    got = _run_sampled(tg, A, B, M, N, K, rows, cols, relu=True)
    want, _ = oracle.gemm_at(A, B, K, rows, cols, relu=True)
    check(got, want, K, relu=True, what=f"{M}x{N}x{K}")


@pytest.fixture(scope="module")
def k_million_inputs():
    M, N, K = 256, 384, 1 << 20
    return M, N, K, W.draw_inputs(M, N, K, ("ints", -1, 2), ("ints", -1, 2), 33)


@pytest.mark.parametrize("cfg", [None, "pair256"])
def test_k_of_a_million(tg, monkeypatch, k_million_inputs, cfg):
    """K = 2^20 on {-1, 0, 1}: the planner's one-CTA 128x64 tiles, and the
    pair kernel (two tiles, each cut into four k-pieces of 262144 k)."""
    if cfg is None:
        monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    else:
        monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    M, N, K, (A, B) = k_million_inputs
    rng = np.random.default_rng(34)
    rows = np.concatenate([rng.integers(0, M, 400), [0, M - 1, 127, 128, 255]]).astype(np.int64)
    cols = np.concatenate([rng.integers(0, N, 400), [N - 1, 0, 63, 64, 383]]).astype(np.int64)
    got = _run_sampled(tg, A, B, M, N, K, rows, cols, relu=False)
    if cfg == "pair256":
        launched = tg.tg_debug_last_launch()
        assert launched.cluster == 2
        if launched.grid == 16:
            assert launched.split_k == 4
    want, _ = oracle.gemm_at(A, B, K, rows, cols)
    check(got, want, K, exact=True, what=f"{M}x{N}x{K} {cfg or 'planned'}")


def test_skinny_n_of_four_million(tg, monkeypatch):
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M, N, K = 64, 1 << 22, 64
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), 35)
    plan = tg.tg_plan_f16(M, N, K, 152)
    assert plan.kernel == tg.TG_KERNEL_SKINNY
    rows, cols = _positions(M, N, 43)
    got = _run_sampled(tg, A, B, M, N, K, rows, cols, relu=False)
    want, _ = oracle.gemm_at(A, B, K, rows, cols)
    check(got, want, K, what=f"{M}x{N}x{K}")
