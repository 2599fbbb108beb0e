"""Parity of the 2:4 structured-sparse GEMM (tg_gemm_sp24, through the C ABI)
against the oracle on a GB300, for both of its kernels (one CTA with 128×128
tiles, and CTA pairs with 256×256 tiles, forced through TGEMM_FORCE_SP24):
ragged shapes (M, N off the tile, K not a multiple of the 128-k stage, a pair
whose second CTA lies wholly past M), fp16 and bf16, the extended epilogue,
integer inputs (exact), the bounded-wait fault path and sampled outputs at the
MLP layer's full size.  Tolerances are those of parity.py and test_gpu_epilogue.py:
the kept values enter the same fp32 accumulation as the dense GEMM."""

import numpy as np
import pytest

import oracle
from exact import bf16_bits_to_float
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


TDT = {"f16": torch.float16, "bf16": torch.bfloat16}
KERNELS = ["cta", "pair"]


@pytest.fixture(params=KERNELS)
def kern(request, monkeypatch):
    """Selects the sparse kernel for the calls of one test."""
    monkeypatch.setenv("TGEMM_FORCE_SP24", request.param)
    return request.param


def to16(x64, fmt):
    t = torch.from_numpy(np.ascontiguousarray(x64, dtype=np.float64)).to(TDT[fmt])
    return t.view(torch.int16).numpy().view(np.uint16)


def dev16(bits, fmt, ld=None):
    rows, cols = bits.shape
    ld = cols if ld is None else ld
    buf = torch.zeros((rows, ld), dtype=torch.int16)
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return buf.cuda().view(TDT[fmt])[:, :cols]


def dev_words(E, ld=None):
    rows, cols = E.shape
    ld = cols if ld is None else ld
    buf = np.zeros((rows, ld), dtype=np.uint32)
    buf[:, :cols] = E
    return torch.from_numpy(buf.view(np.int32)).cuda()[:, :cols]


def decode(bits, fmt):
    if fmt == "bf16":
        return bf16_bits_to_float(bits)
    return np.ascontiguousarray(bits).view(np.float16).astype(np.float64)


def run(tg, fmt, Ac, E, B, M, N, K, *, relu=False, bias=None, R=None, out=None, lde=None):
    out = out or fmt
    ac = dev16(Ac, fmt, ld=W.round16(K // 2) if K else 8)
    e = dev_words(E, ld=lde if lde is not None else max(4, (K // 32 + 3) // 4 * 4))
    b = dev16(B, fmt, ld=max(8, -(-N // 8) * 8))
    dt = torch.float32 if out == "f32" else TDT[fmt]
    c = torch.full((M, -(-N // 8) * 8), float("nan"), dtype=dt, device="cuda")[:, :N]
    bias_d = torch.from_numpy(bias).cuda() if bias is not None else None
    r_d = dev16(R, fmt) if R is not None else None
    in_code = tg.TG_DTYPE_BF16 if fmt == "bf16" else tg.TG_DTYPE_F16
    epi = tg.tg_epilogue_ex_t(1 if relu else 0, tg.TG_DTYPE_F32 if out == "f32" else in_code,
                              bias_d.data_ptr() if bias_d is not None else None,
                              r_d.data_ptr() if r_d is not None else None,
                              N if r_d is not None else 0)
    s = torch.cuda.current_stream().cuda_stream
    st = tg.tg_gemm_sp24(in_code, ac.data_ptr(), e.data_ptr(), b.data_ptr(), c.data_ptr(), M, N,
                         K, ac.stride(0) if M > 1 else W.round16(K // 2), e.stride(0) if M > 1 else
                         max(4, (K // 32 + 3) // 4 * 4), b.stride(0) if K > 1 else
                         max(8, -(-N // 8) * 8), c.stride(0) if M > 1 else -(-N // 8) * 8, epi, s)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_sync_status(s) == tg.TG_OK
    if out == "f32":
        return c.cpu().numpy().astype(np.float64)
    return decode(c.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), fmt)


def case(M, N, K, fmt, seed, integer=False):
    rng = np.random.default_rng([seed, 0])
    dist_a = ("ints", -2, 3) if integer else ("normal", 0.0, 1.0)
    Ac, E = W.draw_sp24(rng, M, K, dist_a)
    Ac = to16(Ac.astype(np.float64), fmt)
    B64 = W.draw(np.random.default_rng([seed, 1]),
                 ("ints", -2, 3) if integer else ("normal", 0.0, 1.0 / np.sqrt(K)), K, N)
    return Ac, E, to16(B64, fmt)


SHAPES = [(128, 128, 128), (1, 64, 32), (129, 200, 96), (300, 1000, 512), (257, 513, 160),
          (1024, 256, 4096)]


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SHAPES])
def test_sp24_parity(tg, kern, M, N, K, fmt):
    Ac, E, B = case(M, N, K, fmt, 1000 + M + N + K)
    for relu in (False, True):
        got = run(tg, fmt, Ac, E, B, M, N, K, relu=relu)
        want = oracle.gemm_sp24(Ac, E, B, M, N, K, relu=relu, in_dtype=fmt)
        check(got, decode(want, fmt) if fmt == "bf16" else want, K, relu=relu, fmt=fmt,
              what=f"sp24 {fmt} {M}x{N}x{K} relu={relu}")


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_sp24_epilogue(tg, kern, fmt):
    M, N, K = 200, 300, 256
    Ac, E, B = case(M, N, K, fmt, 7)
    rng = np.random.default_rng(8)
    bias = rng.normal(0, 0.5, N).astype(np.float32)
    R = to16(rng.normal(0, 1, (M, N)), fmt)
    got = run(tg, fmt, Ac, E, B, M, N, K, relu=True, bias=bias, R=R)
    want = oracle.gemm_sp24(Ac, E, B, M, N, K, relu=True, bias=bias, R=R, in_dtype=fmt)
    check(got, decode(want, fmt) if fmt == "bf16" else want, K, fmt=fmt, what="sp24 epilogue")
    got = run(tg, fmt, Ac, E, B, M, N, K, bias=bias, out="f32")
    want = oracle.gemm_sp24(Ac, E, B, M, N, K, bias=bias, in_dtype=fmt, out_dtype="f32")
    A = decode(oracle.sp24_decompress(Ac, E, M, K), fmt)
    T = np.abs(A) @ np.abs(decode(B, fmt)) + np.abs(bias.astype(np.float64))
    tol = 2.0 * np.spacing(np.abs(want).astype(np.float32)).astype(np.float64) \
        + (K + 2) * 2.0 ** -23 * T
    assert np.all(np.abs(got - want.astype(np.float64)) <= tol), "sp24 f32 out"


@pytest.mark.parametrize("M,N,K", [(256, 384, 1024), (512, 512, 512)])
def test_sp24_integers_exact(tg, kern, M, N, K):
    """Integer kept values and B: every partial sum is an exact integer in fp32,
    so the result equals the oracle exactly (this pins the metadata layout in
    tensor memory, for the pair kernel in both CTAs: a wrong position would
    change some sum)."""
    Ac, E, B = case(M, N, K, "f16", 11, integer=True)
    got = run(tg, "f16", Ac, E, B, M, N, K)
    want = oracle.gemm_sp24(Ac, E, B, M, N, K).astype(np.float64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(2560, 2304, 288), (2304, 2560, 544), (2500, 2300, 288)])
def test_sp24_ring_across_tiles_exact(tg, kern, M, N, K):
    """More 256×256 tiles (90) than CTA pairs fit on the GPU, with 3 and 5
    k blocks of 128: a cluster runs two tiles, and its operand and metadata
    rings carry on from one tile into the next at a stage offset other than 0
    (4-stage plain build, and 3-stage full build through the bias).  Integer
    inputs: every sum is exact, so C equals the oracle bit for bit."""
    Ac, E, B = case(M, N, K, "f16", 15 + K, integer=True)
    got = run(tg, "f16", Ac, E, B, M, N, K)
    assert np.array_equal(got, oracle.gemm_sp24(Ac, E, B, M, N, K).astype(np.float64))
    bias = np.random.default_rng(16 + K).integers(-4, 5, N).astype(np.float32)
    got = run(tg, "f16", Ac, E, B, M, N, K, relu=True, bias=bias)
    want = oracle.gemm_sp24(Ac, E, B, M, N, K, relu=True, bias=bias)
    assert np.array_equal(got, want.astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(512, 512, 8192), (1024, 1024, 1024), (256, 2048, 4096)])
def test_sp24_planner_choice(tg, monkeypatch, M, N, K):
    """The planner's own kernel (no override): long K below a wave takes the
    CTA pairs (512×512×8192, 256×2048×4096), short K the one-CTA kernel (1024³)."""
    monkeypatch.delenv("TGEMM_FORCE_SP24", raising=False)
    Ac, E, B = case(M, N, K, "f16", 17 + M + K)
    got = run(tg, "f16", Ac, E, B, M, N, K, relu=True)
    check(got, oracle.gemm_sp24(Ac, E, B, M, N, K, relu=True), K, relu=True,
          what=f"sp24 planned {M}x{N}x{K}")


def test_sp24_metadata_padding(tg, kern):
    """Metadata words past K/32 in a padded row stride are never used."""
    M, N, K = 64, 128, 96
    Ac, E, B = case(M, N, K, "f16", 12)
    Ep = np.full((M, 8), 0xFFFFFFFF, dtype=np.uint32)  # invalid if read
    Ep[:, :3] = E[:, :3]
    got = run(tg, "f16", Ac, Ep, B, M, N, K, lde=8)
    check(got, oracle.gemm_sp24(Ac, E, B, M, N, K), K, what="sp24 padded metadata")


def test_sp24_withheld_signal_times_out_and_recovers(tg, kern):
    M, N, K = 256, 256, 256
    Ac, E, B = case(M, N, K, "f16", 13)
    s = torch.cuda.current_stream().cuda_stream
    assert tg.tg_sync_status(s) == tg.TG_OK
    try:
        tg.tg_debug_set_wait_timeout_ns(50_000_000)
        tg.tg_debug_inject(1)
        ac, e, b = dev16(Ac, "f16"), dev_words(E, ld=8), dev16(B, "f16")
        c = torch.zeros((M, N), dtype=torch.float16, device="cuda")
        st = tg.tg_gemm_sp24(tg.TG_DTYPE_F16, ac.data_ptr(), e.data_ptr(), b.data_ptr(),
                             c.data_ptr(), M, N, K, K // 2, 8, N, N, None, s)
        assert st == tg.TG_OK
        assert tg.tg_sync_status(s) == tg.TG_ERR_TIMEOUT
        assert tg.tg_sync_status(s) == tg.TG_OK
    finally:
        tg.tg_debug_inject(0)
        tg.tg_debug_set_wait_timeout_ns(0)
    check(run(tg, "f16", Ac, E, B, M, N, K), oracle.gemm_sp24(Ac, E, B, M, N, K), K,
          what="sp24 after timeout")


def test_sp24_python_api(tg):
    M, N, K = 96, 160, 192
    Ac, E, B = case(M, N, K, "f16", 14)
    ac = torch.from_numpy(Ac.view(np.float16)).cuda()
    ebuf = np.zeros((M, 8), dtype=np.uint32)  # row stride a multiple of 4 words
    ebuf[:, :K // 32] = E
    e = torch.from_numpy(ebuf.view(np.int32)).cuda()[:, :K // 32]
    b = torch.from_numpy(B.view(np.float16)).cuda()
    c = tg.gemm_sp24(ac, e, b, relu=True)
    torch.cuda.synchronize()
    check(c.cpu().numpy(), oracle.gemm_sp24(Ac, E, B, M, N, K, relu=True), K, relu=True,
          what="sp24 python api")
    with pytest.raises(ValueError):
        tg.gemm_sp24(ac[:, :-8], e, b)


def test_sp24_mlp_full_size_sampled(tg, kern):
    """8192×28672×4096 with a 2:4 A, as the benchmark runs it (the pair
    kernel) and on the one-CTA kernel: sampled outputs."""
    w = W.SP24_WORKLOADS["sp24_mlp_8192x28672x4096_relu"]
    Ac, E, B = W.sp24_workload_inputs(w)
    ac = torch.from_numpy(Ac).cuda()
    e = torch.from_numpy(E.view(np.int32)).cuda()
    b = torch.from_numpy(B).cuda()
    c = tg.gemm_sp24(ac, e, b, relu=w.relu)
    tg.sync_status()
    rows, cols = W.sample_positions(w.M, w.N, 128, 128, w.seed)
    got = c[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    want, _ = oracle.gemm_sp24_at(Ac.view(np.uint16), E, B.view(np.uint16), w.K, rows, cols,
                                  relu=w.relu)
    check(got, want, w.K, relu=w.relu, what=w.name)
    del ac, e, b, c
    torch.cuda.empty_cache()
