"""tg_gemm_f16_host (C = epi(A·B) with A, B, C in host memory, copies
overlapped with the products block by block) against the oracle on a GB300:
one column block, several with a ragged last one (up to six for wide C), host row strides with
padding (odd ones included: the device copies are re-pitched), M <= 128 (the
split-K kernel per block), K = 0, pageable host memory, and calls of
different sizes back to back on one stream (the device copies grow)."""

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


def host_matrix(x16, ld, pinned=True):
    """A host fp16 buffer rows × ld holding x16 in its first columns (the
    padding set to a marker) and the view of the data."""
    rows, cols = x16.shape
    buf = torch.full((rows, ld), -7.0, dtype=torch.float16)
    if pinned:
        buf = buf.pin_memory()
    buf[:, :cols] = torch.from_numpy(x16)
    return buf


def run(tg, M, N, K, relu, pads=(0, 0, 0), pinned=True, seed=0):
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(max(K, 1))), seed)
    lda, ldb, ldc = K + pads[0], N + pads[1], N + pads[2]
    ha = host_matrix(A, max(lda, 1), pinned)
    hb = host_matrix(B, max(ldb, 1), pinned)
    hc = host_matrix(np.zeros((M, N), np.float16), max(ldc, 1), pinned)
    hc[:, :N] = float("nan")
    s = torch.cuda.current_stream().cuda_stream
    st = tg.tg_gemm_f16_host(ha.data_ptr(), hb.data_ptr(), hc.data_ptr(), M, N, K, max(lda, 1),
                             max(ldb, 1), max(ldc, 1), tg.TG_EPI_RELU if relu else tg.TG_EPI_NONE,
                             s)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_sync_status(s) == tg.TG_OK
    got = hc[:, :N].numpy()
    if ldc > N:  # padding columns of C are never written
        assert np.all(hc[:, N:].numpy() == np.float16(-7.0))
    return A, B, got


CASES = [  # M, N, K, relu, (pad lda, pad ldb, pad ldc)
    (300, 1000, 200, True, (0, 0, 0)),       # one column block
    (512, 9000, 320, False, (0, 0, 0)),      # blocks of 1024, 2048, 4096 and 1832 columns
    (257, 4100, 96, True, (5, 3, 7)),        # odd host strides, ragged everything
    (64, 6000, 512, False, (8, 0, 16)),      # M <= 128: split-K kernel in every block
    (1, 2500, 33, True, (1, 1, 1)),
    (200, 15000, 64, True, (0, 0, 0)),       # 1024, 2048, 4096, 7832 columns
    (96, 29001, 72, False, (3, 5, 1)),       # six blocks, odd strides, a ragged last block
]


@pytest.mark.parametrize("M,N,K,relu,pads", CASES,
                         ids=[f"{m}x{n}x{k}" for m, n, k, _, _ in CASES])
def test_host_entry_matches_oracle(tg, M, N, K, relu, pads):
    A, B, got = run(tg, M, N, K, relu, pads, seed=M + N + K)
    check(got, oracle.gemm(A, B, M, N, K, relu=relu), K, relu=relu,
          what=f"host {M}x{N}x{K}")


def test_host_entry_k0_fills_zero(tg):
    _, _, got = run(tg, 40, 3000, 0, True, (0, 0, 4))
    assert np.all(got == 0) and not np.any(np.signbit(got))


def test_host_entry_pageable_memory(tg):
    A, B, got = run(tg, 200, 2600, 128, False, (0, 0, 0), pinned=False, seed=3)
    check(got, oracle.gemm(A, B, 200, 2600, 128), 128, what="host pageable")


def test_host_entry_back_to_back_sizes(tg):
    """Calls of growing and shrinking sizes on one stream, each checked: the
    device copies grow between calls and later calls reuse them."""
    for i, (M, N, K) in enumerate([(128, 2048, 64), (700, 9000, 300), (96, 3000, 128)]):
        A, B, got = run(tg, M, N, K, i % 2 == 1, seed=10 + i)
        check(got, oracle.gemm(A, B, M, N, K, relu=i % 2 == 1), K, relu=i % 2 == 1,
              what=f"host call {i}")


def test_gemm_host_python_api(tg):
    M, N, K = 333, 5000, 160
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), 21)
    c = tg.gemm_host(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(),
                     relu=True)
    check(c.numpy(), oracle.gemm(A, B, M, N, K, relu=True), K, relu=True, what="gemm_host")
    with pytest.raises(ValueError):
        tg.gemm_host(torch.from_numpy(A), torch.from_numpy(B)[:-1])
