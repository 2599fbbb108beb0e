"""Parity of the MXFP4 weight GEMM (tg_gemm_mxfp4, through the C ABI) against
the oracle on a GB300.

Both paths are covered: the fused split-K kernel (M <= 128, weights decoded
in shared memory) and dequantise-then-GEMM (M > 128, or forced onto each
dense kernel with TGEMM_FORCE_CFG).  Tolerances are those of the fp16 GEMM
(parity.py) and of the extended epilogue (test_gpu_epilogue.py): the
dequantised weights are fp16 numbers, so once they are decoded the product
is the fp16 GEMM.  The decode itself is checked exactly: with A the identity,
C is Bdeq element for element, over every scale byte 0..254 and every code,
and a NaN scale turns its column to NaN.
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


PATHS = [None, "pair256", "persistent256", "persistent128", "persistent64"]  # None: fused kernel for M <= 128


def dev(x: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run(tg, A, Bq, S, M, N, K, *, relu=False, bias=None, R=None, out="f16", lda=None,
        a_offset=0):
    """Call tg_gemm_mxfp4 on device copies; returns C as float64 on the host."""
    lda = K if lda is None else lda
    abuf = torch.zeros(M * lda + a_offset + 8, dtype=torch.float16)
    abuf[a_offset:a_offset + M * lda].view(M, lda)[:, :K] = torch.from_numpy(A)
    a = abuf.cuda()[a_offset:]
    bq, s = dev(Bq), dev(S)
    dt = torch.float32 if out == "f32" else torch.float16
    c = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    bias_d = dev(bias) if bias is not None else None
    r_d = dev(R) if R is not None else None
    epi = tg.tg_epilogue_ex_t(1 if relu else 0,
                              tg.TG_DTYPE_F32 if out == "f32" else tg.TG_DTYPE_F16,
                              bias_d.data_ptr() if bias_d is not None else None,
                              r_d.data_ptr() if r_d is not None else None,
                              N if r_d is not None else 0)
    st = tg.tg_gemm_mxfp4(a.data_ptr(), bq.data_ptr(), s.data_ptr(), c.data_ptr(), M, N, K,
                          lda, Bq.shape[1], S.shape[1], N, epi,
                          torch.cuda.current_stream().cuda_stream)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_sync_status(torch.cuda.current_stream().cuda_stream) == tg.TG_OK
    return c.cpu().numpy().astype(np.float64)


def case(M, N, K, seed, lo=115, hi=125, **kw):
    rng = np.random.default_rng([seed, 0])
    A = rng.normal(0.0, 1.0, (M, K)).astype(np.float16)
    Bq, S = W.draw_mxfp4(np.random.default_rng([seed, 1]), K, N, lo, hi, **kw)
    return A, Bq, S


SHAPES = [(1, 1, 1), (7, 129, 100), (64, 2048, 520), (128, 1000, 333), (96, 4096, 4096)]


@pytest.mark.parametrize("M,N,K", SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SHAPES])
@pytest.mark.parametrize("path", PATHS, ids=lambda p: p or "fused")
def test_mxfp4_every_path(tg, monkeypatch, path, M, N, K):
    if path is not None:
        monkeypatch.setenv("TGEMM_FORCE_CFG", path)
    else:
        monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    A, Bq, S = case(M, N, K, 900 + M + N + K)
    Bd = oracle.mxfp4_dequant(Bq, S, K, N)
    got = run(tg, A, Bq, S, M, N, K)
    want = oracle.gemm_mxfp4(A, Bq, S, M, N, K)
    check(got, want, K, what=f"{path or 'fused'} {M}x{N}x{K}")
    # repeated calls give the same bits (fixed split-K order)
    assert np.array_equal(run(tg, A, Bq, S, M, N, K), got)
    # fused epilogue: bias + ReLU + residual, and fp32 output
    rng = np.random.default_rng(M + N)
    bias = rng.normal(0, 0.5, N).astype(np.float32)
    R = rng.normal(0, 1, (M, N)).astype(np.float16)
    got = run(tg, A, Bq, S, M, N, K, relu=True, bias=bias, R=R)
    want = oracle.gemm_mxfp4(A, Bq, S, M, N, K, relu=True, bias=bias, R=R)
    check(got, want, K, what=f"{path or 'fused'} epilogue")
    got = run(tg, A, Bq, S, M, N, K, out="f32")
    want = oracle.gemm_mxfp4(A, Bq, S, M, N, K, out_dtype="f32").astype(np.float64)
    T = np.abs(A.astype(np.float64)) @ np.abs(Bd.astype(np.float64))
    tol = 2.0 * np.spacing(np.abs(want).astype(np.float32)).astype(np.float64) \
        + (K + 2) * 2.0 ** -23 * T
    assert np.all(np.abs(got - want) <= tol), f"{path or 'fused'} f32 out"


@pytest.mark.parametrize("M,N,K", [(300, 1000, 129), (257, 513, 65)])
def test_mxfp4_large_m_dequant_path(tg, monkeypatch, M, N, K):
    """M > 128 takes the dequantise-then-GEMM path without any override."""
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    A, Bq, S = case(M, N, K, 77)
    check(run(tg, A, Bq, S, M, N, K), oracle.gemm_mxfp4(A, Bq, S, M, N, K), K,
          what=f"dequant path {M}x{N}x{K}")


def _pack(codes: np.ndarray, ld: int) -> np.ndarray:
    """K×N codes into N rows of packed bytes along k (low nibble = even k)."""
    K, N = codes.shape
    out = np.zeros((N, ld), dtype=np.uint8)
    for k in range(K):
        out[:, k // 2] |= (codes[k, :].astype(np.uint8) << (4 * (k % 2))).astype(np.uint8)
    return out


E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


@pytest.mark.parametrize("path", PATHS, ids=lambda p: p or "fused")
def test_mxfp4_decode_every_scale_exact(tg, monkeypatch, path):
    """A = identity (M = K = 128), so C = Bdeq exactly.  Columns take scale
    bytes 0..254 (both decode routes, fp16 subnormals, underflow to zero);
    codes are drawn among those whose value stays finite in fp16 so no
    column holds an infinity (0·inf would turn a whole column to NaN)."""
    if path is not None:
        monkeypatch.setenv("TGEMM_FORCE_CFG", path)
    else:
        monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M = K = 128
    N = 512
    rng = np.random.default_rng(3)
    X = rng.integers(0, 255, size=(K // 32, N)).astype(np.uint8)
    X[:, :255] = np.arange(255, dtype=np.uint8)[None, :]  # every scale byte in some column
    codes = np.zeros((K, N), dtype=np.int64)
    for n in range(N):
        for b in range(K // 32):
            x = int(X[b, n])
            ok = [c for c in range(16) if E2M1_MAG[c & 7] * 2.0 ** (x - 127) < 65520.0]
            codes[32 * b:32 * b + 32, n] = rng.choice(ok, size=32)
    Bq = _pack(codes, W.round16((K + 1) // 2))
    S = np.zeros((K // 32, W.round16(N)), dtype=np.uint8)
    S[:, :N] = X
    A = np.eye(M, K, dtype=np.float16)
    got = run(tg, A, Bq, S, M, N, K)
    want = oracle.mxfp4_dequant(Bq, S, K, N).astype(np.float64)
    assert np.all(np.isfinite(want))
    bad = got != want
    assert not np.any(bad), (f"{int(bad.sum())} decoded weights differ; first "
                             f"{np.argwhere(bad)[:5].tolist()}")


def test_mxfp4_nan_scale(tg, monkeypatch):
    """A NaN scale (255) makes its block NaN, and through A's zeros its whole
    column of C NaN; the other columns stay exact."""
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M = K = 64
    N = 64
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 16, (K, N))
    X = np.full((K // 32, 64), 120, dtype=np.uint8)
    X[1, 5] = 255
    Bq = _pack(codes, 32)  # K = 64: 32 bytes per column
    A = np.eye(M, K, dtype=np.float16)
    got = run(tg, A, Bq, X, M, N, K)
    want = oracle.mxfp4_dequant(Bq, X, K, N).astype(np.float64)
    assert np.all(np.isnan(got[:, 5]))
    keep = np.arange(N) != 5
    assert np.array_equal(got[:, keep], want[:, keep])


@pytest.mark.parametrize("path", [None, "pair256"], ids=["fused", "dequant"])
def test_mxfp4_layouts(tg, monkeypatch, path):
    """Odd K (a spare nibble of random bits), K not a multiple of 32 or 64,
    N not a multiple of 128, padded code and scale rows (random padding), A
    with an odd row stride at an address off 16 bytes (staged)."""
    if path is not None:
        monkeypatch.setenv("TGEMM_FORCE_CFG", path)
    else:
        monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M, N, K = 50, 777, 201
    A, Bq, S = case(M, N, K, 13, ldbq=128, lds=800)
    got = run(tg, A, Bq, S, M, N, K, lda=203, a_offset=1)
    check(got, oracle.gemm_mxfp4(A, Bq, S, M, N, K), K, what=f"layouts {path}")


def test_mxfp4_k0_and_python_api(tg):
    M, N, K = 40, 96, 300
    A, Bq, S = case(M, N, K, 21)
    a, bq, s = dev(A), dev(Bq), dev(S)
    rng = np.random.default_rng(22)
    bias = rng.normal(0, 1, N).astype(np.float32)
    c = tg.gemm_mxfp4(a, bq, s, N, relu=True, bias=dev(bias), out_dtype=torch.float32)
    torch.cuda.synchronize()
    want = oracle.gemm_mxfp4(A, Bq, S, M, N, K, relu=True, bias=bias, out_dtype="f32")
    Bd = oracle.mxfp4_dequant(Bq, S, K, N).astype(np.float64)
    T = np.abs(A.astype(np.float64)) @ np.abs(Bd) + np.abs(bias.astype(np.float64))
    err = np.abs(c.cpu().numpy().astype(np.float64) - want.astype(np.float64))
    assert np.all(err <= 2.0 ** -22 * np.abs(want) + (K + 2) * 2.0 ** -23 * T)
    # K == 0: C = act(bias)
    e = tg.tg_epilogue_ex_t(1, tg.TG_DTYPE_F16, dev(bias).data_ptr(), None, 0)
    c0 = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    st = tg.tg_gemm_mxfp4(None, None, None, c0.data_ptr(), M, N, 0, 0, 16, 96, N, e, None)
    assert st == tg.TG_OK
    torch.cuda.synchronize()
    assert np.array_equal(c0.cpu().numpy().astype(np.float64),
                          np.broadcast_to(np.maximum(bias, 0).astype(np.float16), (M, N))
                          .astype(np.float64))
    with pytest.raises(TypeError):
        tg.gemm_mxfp4(a.to(torch.bfloat16), bq, s, N)
    with pytest.raises(ValueError):
        tg.gemm_mxfp4(a, bq[:-1], s, N)  # one weight column short


@pytest.mark.parametrize("name", ["mxfp4_skinny_64x16384x8192",
                                  "mxfp4_mlp_8192x28672x4096_relu"])
def test_mxfp4_workload_sampled(tg, monkeypatch, name):
    """Full-size launches as the benchmark runs them, checked on sampled
    outputs (random positions plus whole rows and columns on tile edges)."""
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    w = W.MX_WORKLOADS[name]
    A, Bq, S = W.mx_workload_inputs(w)
    a, bq, s = dev(A), dev(Bq), dev(S)
    c = tg.gemm_mxfp4(a, bq, s, w.N, relu=w.relu)
    tg.sync_status()
    bm = w.M if w.M <= 128 else 256
    rows, cols = W.sample_positions(w.M, w.N, bm, 128 if w.M <= 128 else 256, w.seed)
    got = c[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    want, _ = oracle.gemm_mxfp4_at(A, Bq, S, w.K, w.N, rows, cols, relu=w.relu)
    check(got, want, w.K, relu=w.relu, what=name)
    del a, bq, s, c
    torch.cuda.empty_cache()


def test_mxfp4_withheld_signal_times_out_and_recovers(tg, monkeypatch):
    """The fused kernel's bounded waits: with the first "accumulator ready"
    signal withheld (tg_debug_inject) the epilogue gives up after 50 ms, the
    converter, producer and MMA warps stop on the abort flag, and the kernel
    returns; the next call works."""
    monkeypatch.delenv("TGEMM_FORCE_CFG", raising=False)
    M, N, K = 64, 512, 1024
    A, Bq, S = case(M, N, K, 41)
    s = torch.cuda.current_stream().cuda_stream
    assert tg.tg_sync_status(s) == tg.TG_OK
    a, bq, sc = dev(A), dev(Bq), dev(S)
    c = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    try:
        tg.tg_debug_set_wait_timeout_ns(50_000_000)
        tg.tg_debug_inject(1)
        st = tg.tg_gemm_mxfp4(a.data_ptr(), bq.data_ptr(), sc.data_ptr(), c.data_ptr(), M, N, K,
                              K, Bq.shape[1], S.shape[1], N, None, s)
        assert st == tg.TG_OK
        assert tg.tg_sync_status(s) == tg.TG_ERR_TIMEOUT
        assert tg.tg_sync_status(s) == tg.TG_OK
    finally:
        tg.tg_debug_inject(0)
        tg.tg_debug_set_wait_timeout_ns(0)
    check(run(tg, A, Bq, S, M, N, K), oracle.gemm_mxfp4(A, Bq, S, M, N, K), K,
          what="after timeout (mxfp4)")
