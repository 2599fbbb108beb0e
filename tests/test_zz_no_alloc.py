"""tg_gemm_f16_noalloc: the split-K GEMM for M <= 128 with its scratch in a
fixed array inside the library, for callers that cannot allocate device
memory at call time (for instance a service whose own pool allocator owns all
device memory).

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.  It passes both alone in a fresh
process and after the rest of the suite.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from parity import check  # noqa: E402


@pytest.fixture(scope="module")
def tg():
    from tiled_fp16_gemm_gb300 import build
    build.build()
    import tiled_fp16_gemm_gb300 as t
    return t


def _inputs(M, N, K, seed):
    from tiled_fp16_gemm_gb300 import workloads as W
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), seed)
    return torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()


@pytest.mark.parametrize("M,N,K,relu", [(64, 16384, 8192, False), (37, 1000, 3000, True),
                                        (128, 4096, 344, False), (1, 296, 1000, True)])
def test_noalloc_matches_allocating_entry_point(tg, monkeypatch, M, N, K, relu):
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    a, b = _inputs(M, N, K, 1234 + M)
    s = torch.cuda.current_stream().cuda_stream
    epi = tg.TG_EPI_RELU if relu else tg.TG_EPI_NONE
    ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert tg.tg_gemm_f16(a.data_ptr(), b.data_ptr(), ref.data_ptr(), M, N, K, K, N, N, epi,
                          s) == tg.TG_OK
    assert tg.tg_sync_status(s) == tg.TG_OK
    want = ref.cpu().numpy()
    # two calls in a row: the second reuses the array the first left behind
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        st = tg.tg_gemm_f16_noalloc(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, K, N,
                                    N, epi, s)
        assert st == tg.TG_OK, tg.tg_status_string(st)
        assert tg.tg_sync_status(s) == tg.TG_OK
        check(out.cpu().numpy(), want, K, relu=relu, what=f"noalloc call {call}")


def test_noalloc_rejects_sizes_beyond_its_kernel(tg):
    a, b = _inputs(129, 256, 64, 5)
    c = torch.empty((129, 256), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = tg.tg_gemm_f16_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), 129, 256, 64, 64, 256,
                                256, 0, s)
    assert st == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_sync_status(s) == tg.TG_OK
