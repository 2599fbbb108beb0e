"""The bounded-wait fault path on a GB300, without faulting the GPU.

tg_debug_inject(1) makes the next launch withhold its first "accumulator
ready" signal, so the epilogue's wait runs out (after a 50 ms limit set with
tg_debug_set_wait_timeout_ns).  The kernel must drain what it has in flight,
free its tensor memory and return; tg_sync_status must then report
TG_ERR_TIMEOUT once, and the next ordinary call must work and be correct.
"""

import pytest

import oracle
from parity import check

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    from tiled_fp16_gemm_gb300 import build
    build.build()
    import tiled_fp16_gemm_gb300 as t
    return t


CASES = [("pair256", 512, 512, 256), ("persistent256", 256, 512, 256),
         ("persistent128", 256, 256, 128), ("persistent64", 256, 128, 128),
         ("skinny", 64, 256, 1024)]


@pytest.mark.parametrize("cfg,M,N,K", CASES, ids=[c[0] for c in CASES])
def test_withheld_signal_times_out_and_recovers(tg, monkeypatch, cfg, M, N, K):
    from tiled_fp16_gemm_gb300 import workloads as W
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    A, B = W.draw_inputs(M, N, K, ("uniform", -1, 1), ("uniform", -1, 1), 31 + M)
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    c = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert tg.tg_sync_status(s) == tg.TG_OK
    try:
        tg.tg_debug_set_wait_timeout_ns(50_000_000)
        tg.tg_debug_inject(1)
        st = tg.tg_gemm_f16(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, K, N, N, 0, s)
        assert st == tg.TG_OK  # the launch itself succeeds
        assert tg.tg_sync_status(s) == tg.TG_ERR_TIMEOUT
        assert tg.tg_sync_status(s) == tg.TG_OK  # reported once, then cleared
    finally:
        tg.tg_debug_inject(0)
        tg.tg_debug_set_wait_timeout_ns(0)
    # the injection applied to one launch only; the context is still usable
    st = tg.tg_gemm_f16(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, K, N, N, 0, s)
    assert st == tg.TG_OK
    assert tg.tg_sync_status(s) == tg.TG_OK
    check(c.cpu().numpy(), oracle.gemm(A, B, M, N, K), K, what=f"after timeout ({cfg})")
