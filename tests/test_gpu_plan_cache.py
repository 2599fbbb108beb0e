"""The planner's shape is the launched shape, and the tensor-map cache never
serves a stale map (GPU).

* For a sweep of shapes covering every dense kernel, tg_plan_f16_limits with
  the current device's limits equals what tg_gemm_f16 launched (kernel,
  tiles, grid, k-pieces, column halves, cluster size), read back with
  tg_debug_last_launch.
* Repeated calls reuse their tensor maps (cache hits, no new encodings); a
  changed pointer, a changed leading dimension and new contents behind the
  same pointers each give the oracle's product for the new operands.
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


SHAPES = [
    (8192, 28672, 4096),   # pair kernel, full waves + tail in column halves
    (4096, 4096, 4096),    # pair kernel, tail tiles in column halves
    (512, 512, 16384),     # pair kernel below one wave, tiles in 4 k-pieces
    (2048, 2048, 4096),    # pair kernel below one wave
    (2048, 2048, 512),     # one-CTA 128x128 (short K)
    (1024, 1024, 1024),    # one-CTA 128x64
    (1536, 1024, 1024),    # one-CTA 128x128
    (3000, 2000, 700),     # one-CTA, ragged
    (64, 16384, 8192),     # skinny, whole tiles
    (64, 4096, 4096),      # skinny, four-piece clusters
    (128, 4096, 14336),    # skinny Mp = 128, four-piece clusters
    (37, 1000, 3000),      # skinny, balanced split
    (1, 296, 1000),        # skinny, M = 1
    (300, 200, 0),         # K = 0: fill
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_launch_matches_plan(tg, monkeypatch, M, N, K):
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    monkeypatch.delenv("TGEMM_GROUP_M", raising=False)
    sms, pairs, qn, qw = tg.tg_device_limits()
    assert sms == torch.cuda.get_device_properties(0).multi_processor_count
    assert 1 <= pairs <= sms // 2 and qn >= 0 and qw >= 0
    want = tg.tg_plan_f16_limits(M, N, K, sms, pairs, qn, qw)
    a = torch.randn(M, max(K, 1), device="cuda").half()[:, :K]
    b = torch.randn(max(K, 1), N, device="cuda").half()[:K]
    c = tg.gemm(a.contiguous(), b.contiguous())
    tg.sync_status()
    got = tg.tg_debug_last_launch()
    for f in ("kernel", "bm", "bn", "bk", "stages", "tiles_m", "tiles_n", "k_blocks",
              "num_tiles", "grid", "split_k", "cluster", "split_n"):
        assert getattr(got, f) == getattr(want, f), (f, getattr(got, f), getattr(want, f))
    del a, b, c


def _dev(x16, ld=None):
    rows, cols = x16.shape
    ld = cols if ld is None else ld
    buf = torch.full((rows, ld), float("nan"), dtype=torch.float16)
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(x16))
    return buf.cuda()


def _call(tg, a, b, c, M, N, K):
    s = torch.cuda.current_stream().cuda_stream
    st = tg.tg_gemm_f16(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, a.stride(0),
                        b.stride(0), c.stride(0), 0, s)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_sync_status(s) == tg.TG_OK
    return c[:, :N].cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(300, 500, 400), (64, 3000, 2048), (2048, 2048, 1024)])
def test_map_cache_reuse(tg, monkeypatch, M, N, K):
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    A, B = W.draw_inputs(M, N, K, ("uniform", -1, 1), ("uniform", -1, 1), 600 + M)
    A2, B2 = W.draw_inputs(M, N, K, ("uniform", -1, 1), ("uniform", -1, 1), 700 + M)
    a, b = _dev(A), _dev(B)
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    check(_call(tg, a, b, c, M, N, K), oracle.gemm(A, B, M, N, K), K, what="first call")

    # the same call again: every map from the cache
    h0, m0 = tg.tg_debug_map_cache_stats()
    check(_call(tg, a, b, c, M, N, K), oracle.gemm(A, B, M, N, K), K, what="repeat")
    h1, m1 = tg.tg_debug_map_cache_stats()
    assert m1 == m0 and h1 >= h0 + 2  # A and B (and C on the tile kernels)

    # a changed B pointer (other data): the new product.  (Whether its map is
    # a hit depends on the allocator: an address and shape seen before in
    # this process gives the same map, which is then correct to reuse.)
    b2 = _dev(B2)
    check(_call(tg, a, b2, c, M, N, K), oracle.gemm(A, B2, M, N, K), K, what="new B pointer")

    # a changed leading dimension of A (still 16-byte rows: no staging)
    a_ld = _dev(A, K + 8)
    check(_call(tg, a_ld, b, c, M, N, K), oracle.gemm(A, B, M, N, K), K, what="new lda")

    # new contents behind the first pointers: the cached maps read them
    a.copy_(torch.from_numpy(A2).cuda())
    b.copy_(torch.from_numpy(B2).cuda())
    check(_call(tg, a, b, c, M, N, K), oracle.gemm(A2, B2, M, N, K), K, what="new contents")
