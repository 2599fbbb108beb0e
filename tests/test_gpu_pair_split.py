"""Parity of the CTA-pair kernel where it cuts its last wave of tiles.

With T tiles on P pairs, the R = T mod P tiles of the last, partial wave are
shared out to otherwise idle pairs in one of two ways (tile_schedule.h):
  - two column halves per tile, each a 256×128 product over all of k (an
    N = 128 pair MMA on one 64-column box of B per CTA), no partial sums;
  - for long k only, up to 4 k-pieces per tile (each at least 1024 k), whose
    fp32 partials are summed in k order by the piece that finishes last.
The cases (at 76 pairs):
  512×512×16384    4 tiles: 4 k-pieces each, 16 pairs;
  300×700×12288    6 tiles, ragged edges: 4 k-pieces each, 24 pairs;
  300×700×2048     6 tiles, ragged: column halves, 12 pairs;
  1280×1500×1024   30 tiles: column halves, 60 pairs; the last column
                   block's right half holds 92 of its 128 columns;
  1200×1300×2048   30 tiles, ragged rows: the last column block's right half
                   lies wholly beyond N (loads read zeros, stores are skipped);
  2560×2048×4096   80 tiles: one full wave, then 4 tiles in column halves
                   (the planner's own choice, asserted);
  4096×4096×1024   256 tiles: three waves, then 28 tiles in column halves
                   (the planner's choice, asserted).
Expected values come from the oracle; the tolerance is parity.py's.  On
{-1, 0, 1} inputs every partial sum is an integer, exact in fp32 in any
grouping, so there the result must equal the oracle exactly.
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


# (M, N, K, forced config or None for the planner's, (split_k, split_n) expected)
CASES = [(512, 512, 16384, "pair256", (4, 1)), (300, 700, 12288, "pair256", (4, 1)),
         (300, 700, 2048, "pair256", (1, 2)), (1280, 1500, 1024, "pair256", (1, 2)),
         (1200, 1300, 2048, "pair256", (1, 2)), (2560, 2048, 4096, None, (1, 2)),
         (4096, 4096, 1024, None, (1, 2))]


def _gemm(tg, A, B, relu=False):
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    c = tg.gemm(a, b, relu=relu)
    tg.sync_status()
    return c.cpu().numpy()


@pytest.mark.parametrize("M,N,K,cfg,cuts", CASES,
                         ids=[f"{m}x{n}x{k}" for m, n, k, _, _ in CASES])
@pytest.mark.parametrize("relu", [False, True])
def test_split_tail_parity(tg, monkeypatch, M, N, K, cfg, cuts, relu):
    if cfg is None:
        monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
        plan = tg.tg_plan_f16(M, N, K, 152)
        assert plan.cluster == 2 and plan.grid == 152
    else:
        monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), M + N + K)
    C = _gemm(tg, A, B, relu)
    launched = tg.tg_debug_last_launch()
    if launched.grid == 152:  # all 76 pairs resident on this device: the cuts above
        assert (launched.split_k, launched.split_n) == cuts, (M, N, K)
    check(C, oracle.gemm(A, B, M, N, K, relu=relu), K, relu=relu, what=f"split {M}x{N}x{K}")
    # the summation order is fixed by the sizes: the same bits on a second call
    assert np.array_equal(_gemm(tg, A, B, relu).view(np.uint16), C.view(np.uint16))


@pytest.mark.parametrize("M,N,K", [(512, 768, 2048), (256, 512, 12288)],
                         ids=["column-halves", "k-pieces"])
def test_split_tail_exact_integers(tg, monkeypatch, M, N, K):
    """Tail tiles in column halves (6 tiles) and in 4 k-pieces (2 tiles) on
    {-1, 0, 1} inputs: exact."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", "pair256")
    A, B = W.draw_inputs(M, N, K, ("ints", -1, 2), ("ints", -1, 2), 4242)
    check(_gemm(tg, A, B), oracle.gemm(A, B, M, N, K), K, exact=True, what="split ints")
    check(_gemm(tg, A, B, relu=True), oracle.gemm(A, B, M, N, K, relu=True), K, exact=True,
          relu=True, what="split ints relu")


def test_column_halves_4096_cubed(tg, monkeypatch):
    """The 4096^3 shape as planned (28 tail tiles in column halves), checked on
    sampled elements plus whole rows and columns at every 128 boundary edge
    of the first, middle and last tiles, which include the tail tiles'
    halves (columns 3584-4095)."""
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M = N = K = 4096
    plan = tg.tg_plan_f16(M, N, K, 152)
    assert plan.split_n == 2 and plan.split_k == 1
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), 4096)
    C = _gemm(tg, A, B, relu=True)
    rows, cols = W.sample_positions(M, N, 128, 128, 11)
    want, _ = oracle.gemm_at(A, B, K, rows, cols, relu=True)
    check(C[rows, cols], want, K, relu=True, what="4096^3 column halves")


def test_split_tail_graph_replay(tg, monkeypatch):
    """A split launch captured in a CUDA graph after one eager call on the
    stream: its partial slots and counters exist, and every replay leaves the
    counters at zero for the next one."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", "pair256")
    M, N, K = 256, 512, 16384  # 2 tiles in 4 k-pieces each
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), 77)
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    s = torch.cuda.Stream()
    eager = torch.empty((M, N), dtype=torch.float16, device="cuda")
    graphed = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    with torch.cuda.stream(s):
        tg.gemm(a, b, out=eager, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tg.gemm(a, b, out=graphed, stream=torch.cuda.current_stream())
    for _ in range(3):
        graphed.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(graphed.view(torch.int16), eager.view(torch.int16))
    assert tg.tg_sync_status(s.cuda_stream) == tg.TG_OK
    check(eager.cpu().numpy(), oracle.gemm(A, B, M, N, K), K, what="split graph")
