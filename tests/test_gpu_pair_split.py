"""Parity of the CTA-pair kernel where it splits its last wave of tiles along k.

With T tiles on P pairs, the R = T mod P tiles of the last, partial wave are
cut into S k-pieces (up to 4, each at least 1024 k long) run by otherwise
idle pairs; their fp32 partials are summed in k order by the piece that
finishes last.  The cases (at 76 pairs):
  512×512×4096     4 tiles: 4 pieces each, 16 pairs;
  1000×1000×8192   16 tiles, ragged edges: 4 pieces each, 64 pairs;
  300×700×2048     6 tiles, ragged: 2 pieces each (K allows two), 12 pairs;
  2560×2048×4096   80 tiles: one full wave, then 4 tiles in 4 pieces each
                   (the planner's own choice, asserted).
Expected values come from the oracle; the tolerance is parity.py's.  On
{-1, 0, 1} inputs every partial sum is an integer, exact in fp32 in any
grouping, so there the split result must equal the oracle exactly.
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


CASES = [(512, 512, 4096, "pair256"), (1000, 1000, 8192, "pair256"),
         (300, 700, 2048, "pair256"), (2560, 2048, 4096, None)]


def _gemm(tg, A, B, relu=False):
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    c = tg.gemm(a, b, relu=relu)
    tg.sync_status()
    return c.cpu().numpy()


@pytest.mark.parametrize("M,N,K,cfg", CASES, ids=[f"{m}x{n}x{k}" for m, n, k, _ in CASES])
@pytest.mark.parametrize("relu", [False, True])
def test_split_tail_parity(tg, monkeypatch, M, N, K, cfg, relu):
    if cfg is None:
        monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
        plan = tg.tg_plan_f16(M, N, K, 152)
        assert plan.cluster == 2 and plan.split_k == 4 and plan.grid == 152
    else:
        monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), M + N + K)
    C = _gemm(tg, A, B, relu)
    check(C, oracle.gemm(A, B, M, N, K, relu=relu), K, relu=relu, what=f"split {M}x{N}x{K}")
    # the summation order is fixed by the sizes: the same bits on a second call
    assert np.array_equal(_gemm(tg, A, B, relu).view(np.uint16), C.view(np.uint16))


def test_split_tail_exact_integers(tg, monkeypatch):
    """6 tiles in 2 pieces each on {-1, 0, 1} inputs: exact."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", "pair256")
    M, N, K = 512, 768, 2048
    A, B = W.draw_inputs(M, N, K, ("ints", -1, 2), ("ints", -1, 2), 4242)
    check(_gemm(tg, A, B), oracle.gemm(A, B, M, N, K), K, exact=True, what="split ints")
    check(_gemm(tg, A, B, relu=True), oracle.gemm(A, B, M, N, K, relu=True), K, exact=True,
          relu=True, what="split ints relu")


def test_split_tail_graph_replay(tg, monkeypatch):
    """A split launch captured in a CUDA graph after one eager call on the
    stream: its partial slots and counters exist, and every replay leaves the
    counters at zero for the next one."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", "pair256")
    M, N, K = 512, 512, 4096
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
