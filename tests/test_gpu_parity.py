"""Parity of libtgemm (through its C ABI) against the CPU oracle on a GB300.

Every input comes from the seeded generators in tiled_fp16_gemm_gb300.workloads
and every expected value from oracle/ (never from the CUDA path).
"""

import numpy as np
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


from tiled_fp16_gemm_gb300 import workloads as W  # noqa: E402


def dev_matrix(x16: np.ndarray, ld: int | None = None, fill=0.0):
    """Copy a float16 (rows×cols) array to the GPU as a row-major view with row
    stride ld (padding columns set to `fill`)."""
    rows, cols = x16.shape
    ld = cols if ld is None else ld
    buf = torch.full((rows, max(ld, 1)), fill, dtype=torch.float16)
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(x16))
    return buf.cuda()[:, :cols]


def run(tg, A16, B16, M, N, K, relu=False, lda=None, ldb=None, ldc=None, c_fill=None):
    """C = epi(A·B) through tg_gemm_f16; returns (C as numpy fp16, device buffer)."""
    a = dev_matrix(A16[:, :K], lda, np.nan)
    b = dev_matrix(B16[:, :N], ldb, np.nan)
    ldc = N if ldc is None else ldc
    cbuf = torch.full((M, max(ldc, 1)), np.nan if c_fill is None else c_fill,
                      dtype=torch.float16, device="cuda")
    c = cbuf[:, :N]
    s = torch.cuda.current_stream()
    st = tg.tg_gemm_f16(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                        a.stride(0) if M > 1 else max(8, -(-K // 8) * 8),
                        b.stride(0) if K > 1 else max(8, -(-N // 8) * 8),
                        cbuf.stride(0) if M > 1 else max(8, -(-N // 8) * 8),
                        1 if relu else 0, s.cuda_stream)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_sync_status(s.cuda_stream) == tg.TG_OK
    return c.cpu().numpy(), cbuf


def ld8(x):
    return max(8, -(-x // 8) * 8)


# ---------------------------------------------------------------- first: one tile

CFGS = ["pair256", "persistent256", "persistent128", "persistent64", "skinny"]


@pytest.fixture(params=CFGS)
def forced(request, monkeypatch):
    monkeypatch.setenv("TGEMM_FORCE_CFG", request.param)
    return request.param


def test_00_single_tile_identity(tg, monkeypatch):
    """Two 128-row tiles, one k step: C = A·I must reproduce A exactly."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", "persistent128")
    M, N, K = 256, 64, 64
    rng = np.random.default_rng(0)
    A = rng.uniform(-2, 2, (M, K)).astype(np.float16)
    I = np.eye(K, N, dtype=np.float16)
    C, _ = run(tg, A, I, M, N, K)
    check(C, A[:, :N], K, exact=True, what="A·I")


def test_01_single_tile_random(tg, forced):
    M, N, K = 128, 256, 64
    A, B = W.draw_inputs(M, N, K, ("uniform", -1, 1), ("uniform", -1, 1), 101)
    C, _ = run(tg, A, B, M, N, K)
    check(C, oracle.gemm(A, B, M, N, K), K, what="128x256x64 " + forced)


def test_02_skinny_single_tile(tg):
    M, N, K = 16, 128, 64
    A, B = W.draw_inputs(M, N, K, ("uniform", -1, 1), ("uniform", -1, 1), 102)
    C, _ = run(tg, A, B, M, N, K)
    check(C, oracle.gemm(A, B, M, N, K), K, what="skinny 16x128x64")


# ---------------------------------------------------------------- the workloads

@pytest.mark.parametrize("name", ["gemm_256", "gemm_1024_relu"])
def test_workload_full(tg, name):
    w = W.WORKLOADS[name]
    A, B = W.workload_inputs(w)
    C, _ = run(tg, A, B, w.M, w.N, w.K, relu=w.relu)
    check(C, oracle.gemm(A, B, w.M, w.N, w.K, relu=w.relu), w.K, relu=w.relu, what=name)


def test_workload_exact_integers(tg):
    w = W.WORKLOADS["gemm_1024_relu_int"]
    A, B = W.workload_inputs(w)
    C, _ = run(tg, A, B, w.M, w.N, w.K, relu=w.relu)
    check(C, oracle.gemm(A, B, w.M, w.N, w.K, relu=w.relu), w.K, exact=True, relu=True,
          what=w.name)
    # the same without ReLU, and through the skinny path (M <= 128)
    C2, _ = run(tg, A, B, w.M, w.N, w.K)
    check(C2, oracle.gemm(A, B, w.M, w.N, w.K), w.K, exact=True, what="ints no relu")
    C3, _ = run(tg, A[:100], B, 100, w.N, w.K)
    check(C3, oracle.gemm(A[:100], B, 100, w.N, w.K), w.K, exact=True, what="ints skinny")


@pytest.mark.parametrize("name", ["gemm_4096", "mlp_8192x28672x4096_relu",
                                  "skinny_64x16384x8192"])
def test_workload_sampled(tg, name):
    """Full-size launch as the benchmark runs it; checked on 4096 random
    elements plus whole rows and columns on tile edges."""
    w = W.WORKLOADS[name]
    A, B = W.workload_inputs(w)
    plan = tg.tg_plan_f16(w.M, w.N, w.K, torch.cuda.get_device_properties(0).multi_processor_count)
    bm = plan.bm if plan.kernel == tg.TG_KERNEL_PERSISTENT else w.M
    bn = plan.bn
    rows, cols = W.sample_positions(w.M, w.N, bm, bn, w.seed)
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    c = tg.gemm(a, b, relu=w.relu)
    tg.sync_status()
    got = c[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    want, _ = oracle.gemm_at(A, B, w.K, rows, cols, relu=w.relu)
    check(got, want, w.K, relu=w.relu, what=name)
    del a, b, c
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- shapes and edges

RAGGED = [(1, 1, 1), (7, 7, 7), (127, 129, 200), (129, 127, 1000), (200, 1000, 129),
          (1000, 200, 7), (129, 1, 127), (200, 7, 1000), (1000, 129, 1), (257, 513, 65),
          (300, 1000, 1000), (129, 2000, 64)]


@pytest.mark.parametrize("M,N,K", RAGGED, ids=[f"{m}x{n}x{k}" for m, n, k in RAGGED])
@pytest.mark.parametrize("relu", [False, True])
def test_ragged_shapes(tg, M, N, K, relu, forced):
    A, B = W.draw_inputs(M, N, K, ("uniform", -1, 1), ("uniform", -1, 1), M * 7 + N * 3 + K)
    C, _ = run(tg, A, B, M, N, K, relu=relu, lda=ld8(K), ldb=ld8(N), ldc=ld8(N))
    check(C, oracle.gemm(A, B, M, N, K, relu=relu), K, relu=relu, what=f"{M}x{N}x{K}")


# (64, 4096, 4096) and (128, 4096, 8192): 32 tiles in 4 equal k pieces on 128 CTAs,
# launched as clusters of a tile's 4 pieces; (16, 14336, 4096): 112 CTAs of one whole tile
# each (the aligned grids); the rest split units evenly
SKINNY = [(1, 300, 1000), (128, 4096, 333), (17, 129, 64), (64, 1000, 1000), (100, 8, 5000),
          (33, 2048, 4096), (64, 16384, 256), (128, 128, 8192), (5, 17, 13), (64, 4096, 4096),
          (16, 14336, 4096), (128, 4096, 8192)]


@pytest.mark.parametrize("M,N,K", SKINNY, ids=[f"{m}x{n}x{k}" for m, n, k in SKINNY])
def test_skinny_shapes(tg, M, N, K):
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), M + N + K)
    C, _ = run(tg, A, B, M, N, K, lda=ld8(K), ldb=ld8(N), ldc=ld8(N))
    check(C, oracle.gemm(A, B, M, N, K), K, what=f"skinny {M}x{N}x{K}")
    Cr, _ = run(tg, A, B, M, N, K, relu=True, lda=ld8(K), ldb=ld8(N), ldc=ld8(N))
    check(Cr, oracle.gemm(A, B, M, N, K, relu=True), K, relu=True, what="skinny relu")


def test_leading_dims_and_padding_untouched(tg):
    M, N, K = 300, 200, 150
    A, B = W.draw_inputs(M, N, K, ("uniform", -1, 1), ("uniform", -1, 1), 55)
    sentinel = 1234.0
    C, cbuf = run(tg, A, B, M, N, K, lda=K + 42, ldb=N + 56, ldc=N + 24, c_fill=sentinel)
    check(C, oracle.gemm(A, B, M, N, K), K, what="padded lds")
    pad = cbuf[:, N:].cpu().numpy().astype(np.float64)
    assert np.all(pad == np.float64(np.float16(sentinel)))
    # skinny path too
    C2, cbuf2 = run(tg, A[:40], B, 40, N, K, lda=K + 42, ldb=N + 56, ldc=N + 24, c_fill=sentinel)
    check(C2, oracle.gemm(A[:40], B, 40, N, K), K, what="skinny padded lds")
    assert np.all(cbuf2[:, N:].cpu().numpy().astype(np.float64) == np.float64(np.float16(sentinel)))


def test_k_zero_and_empty(tg):
    M, N = 37, 45
    cbuf = torch.full((M, 48), 7.0, dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert tg.tg_gemm_f16(0, 0, cbuf.data_ptr(), M, N, 0, 0, 0, 48, 1, s) == tg.TG_OK
    assert tg.tg_sync_status(s) == tg.TG_OK
    out = cbuf.cpu().numpy().astype(np.float64)
    assert np.all(out[:, :N] == 0.0) and not np.any(np.signbit(out[:, :N]))
    assert np.all(out[:, N:] == 7.0)
    before = cbuf.clone()
    assert tg.tg_gemm_f16(0, 0, cbuf.data_ptr(), 0, N, 5, 8, 48, 48, 0, s) == tg.TG_OK
    assert tg.tg_gemm_f16(0, 0, cbuf.data_ptr(), M, 0, 5, 8, 8, 48, 0, s) == tg.TG_OK
    torch.cuda.synchronize()
    assert torch.equal(before, cbuf)


def test_streams_repeat_and_determinism(tg):
    """Two non-default streams, repeated launches: identical bits every time
    (the split-K reduction order is fixed)."""
    shapes = [(64, 4096, 4096, False), (512, 768, 2048, True)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for (M, N, K, relu) in shapes:
        A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 0.02), 77 + M)
        a = torch.from_numpy(A).cuda()
        b = torch.from_numpy(B).cuda()
        torch.cuda.synchronize()
        outs = []
        for i in range(6):
            s = s1 if i % 2 == 0 else s2
            with torch.cuda.stream(s):
                outs.append(tg.gemm(a, b, relu=relu, stream=s))
        torch.cuda.synchronize()
        for o in outs[1:]:
            assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
        check(outs[0].cpu().numpy(), oracle.gemm(A, B, M, N, K, relu=relu), K, relu=relu,
              what=f"streams {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(2048, 9728, 1024), (64, 8192, 4096), (300, 496, 200)],
                         ids=["pair", "skinny", "small"])
def test_cuda_graph_capture_and_replay(tg, M, N, K):
    """tg_gemm_f16 captured in a CUDA graph (after one call on the stream
    outside capture) replays to the same bits as the eager call."""
    A, B = W.draw_inputs(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), 61 + M)
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    s = torch.cuda.Stream()
    eager = torch.empty((M, N), dtype=torch.float16, device="cuda")
    graphed = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    with torch.cuda.stream(s):
        tg.gemm(a, b, relu=True, out=eager, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tg.gemm(a, b, relu=True, out=graphed, stream=torch.cuda.current_stream())
    for _ in range(3):
        graphed.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(graphed.view(torch.int16), eager.view(torch.int16))
    assert tg.tg_sync_status(s.cuda_stream) == tg.TG_OK
    check(eager.cpu().numpy(), oracle.gemm(A, B, M, N, K, relu=True), K, relu=True,
          what="graph")


def test_torch_matmul_sanity(tg):
    """Secondary check (never the product path): agrees with torch's fp16 matmul."""
    M, N, K = 1024, 1536, 768
    a = (torch.randn(M, K, device="cuda") * 0.5).half()
    b = (torch.randn(K, N, device="cuda") * 0.05).half()
    c = tg.gemm(a, b)
    ref = (a.float() @ b.float()).half()
    assert torch.allclose(c.float(), ref.float(), rtol=2e-3, atol=2e-3)


def test_python_api_errors(tg):
    # row stride 6 is not a multiple of 8: accepted through the staging copy
    A, B = W.draw_inputs(4, 8, 6, ("uniform", -1, 1), ("uniform", -1, 1), 3)
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    check(tg.gemm(a, b).cpu().numpy(), oracle.gemm(A, B, 4, 8, 6), 6, what="stride 6")
    with pytest.raises(TypeError):
        tg.gemm(a.float(), b)
    with pytest.raises(ValueError):
        tg.gemm(torch.zeros((4, 8), dtype=torch.float16, device="cuda"), b)


def test_gemm_host_end_to_end(tg):
    M, N, K = 256, 384, 320
    A, B = W.draw_inputs(M, N, K, ("uniform", -1, 1), ("uniform", -1, 1), 9)
    c = tg.gemm_host(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(),
                     relu=True)
    assert not c.is_cuda
    check(c.numpy(), oracle.gemm(A, B, M, N, K, relu=True), K, relu=True, what="gemm_host")
