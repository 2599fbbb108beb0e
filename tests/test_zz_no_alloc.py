"""tg_gemm_f16_noalloc: the split-K GEMM for M <= 128 with its scratch in a
fixed array inside the library, for callers that cannot allocate device
memory at call time (for instance a service whose own pool allocator owns all
device memory).

Each call is checked two ways: against the CPU oracle (full C on the small
shapes, sampled elements plus whole tile-edge rows and columns on the
64x16384x8192 weight-streaming shape, exact equality on {-1, 0, 1} inputs),
and bit for bit against tg_gemm_f16 on the same inputs, which runs the same
kernel with the same plan and the same fixed order of the split-K sum.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.  It passes both alone in a fresh
process and after the rest of the suite.
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


def _expected(A, B, M, N, K, relu):
    """(rows, cols, oracle values): every element when the oracle finishes in
    about a second, else the sampled positions of a 128-column tiling."""
    if M * N * K <= 2 ** 33:
        rows, cols = np.divmod(np.arange(M * N, dtype=np.int64), N)
        return rows, cols, oracle.gemm(A, B, M, N, K, relu=relu).reshape(-1)
    rows, cols = W.sample_positions(M, N, M, 128, 77)
    want, _ = oracle.gemm_at(A, B, K, rows, cols, relu=relu)
    return rows, cols, want


def _run_both(tg, A, B, M, N, K, relu, exact=False):
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    s = torch.cuda.current_stream().cuda_stream
    epi = tg.TG_EPI_RELU if relu else tg.TG_EPI_NONE
    ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert tg.tg_gemm_f16(a.data_ptr(), b.data_ptr(), ref.data_ptr(), M, N, K, K, N, N, epi,
                          s) == tg.TG_OK
    assert tg.tg_sync_status(s) == tg.TG_OK
    same_kernel = ref.cpu().numpy()
    rows, cols, want = _expected(A, B, M, N, K, relu)
    # two calls in a row: the second reuses the array the first left behind
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        st = tg.tg_gemm_f16_noalloc(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, K, N,
                                    N, epi, s)
        assert st == tg.TG_OK, tg.tg_status_string(st)
        assert tg.tg_sync_status(s) == tg.TG_OK
        got = out.cpu().numpy()
        check(got[rows, cols], want, K, exact=exact, relu=relu,
              what=f"noalloc {M}x{N}x{K} call {call} vs oracle")
        assert np.array_equal(got.view(np.uint16), same_kernel.view(np.uint16)), \
            f"noalloc {M}x{N}x{K} call {call}: bits differ from tg_gemm_f16"


@pytest.mark.parametrize("M,N,K,relu", [(64, 16384, 8192, False), (37, 1000, 3000, True),
                                        (128, 4096, 344, False), (1, 296, 1000, True)])
def test_noalloc_matches_oracle_and_allocating_entry_point(tg, monkeypatch, M, N, K, relu):
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), 1234 + M)
    _run_both(tg, A, B, M, N, K, relu)


def test_noalloc_exact_integers(tg, monkeypatch):
    """{-1, 0, 1} inputs with K <= 2048: every partial sum is an exact integer,
    so the split-K result must equal the oracle exactly."""
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M, N, K = 100, 3000, 2048
    A, B = W.draw_inputs(M, N, K, ("ints", -1, 2), ("ints", -1, 2), 4321)
    _run_both(tg, A, B, M, N, K, relu=True, exact=True)


def test_noalloc_rejects_sizes_beyond_its_kernel(tg):
    A, B = W.draw_inputs(129, 256, 64, ("uniform", -1, 1), ("uniform", -1, 1), 5)
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c = torch.empty((129, 256), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = tg.tg_gemm_f16_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), 129, 256, 64, 64, 256,
                                256, 0, s)
    assert st == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_sync_status(s) == tg.TG_OK
