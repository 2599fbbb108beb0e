"""Parity of the bfloat16 variant (tg_gemm_bf16, through the C ABI) against
the oracle's bfloat16 GEMM on a GB300: every kernel, ragged shapes, the
exactness variant and the MLP workload shape."""

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


def bf16_bits(x64: np.ndarray) -> np.ndarray:
    """A float64 matrix as bfloat16 bit patterns (uint16), rounded by torch."""
    t = torch.from_numpy(np.ascontiguousarray(x64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def draw_bf16(M, N, K, dist_a, dist_b, seed):
    a = W.draw(np.random.default_rng([seed, 0]), dist_a, M, K)
    b = W.draw(np.random.default_rng([seed, 1]), dist_b, K, N)
    return bf16_bits(a), bf16_bits(b)


def to_dev(bits: np.ndarray, ld: int | None = None):
    rows, cols = bits.shape
    ld = cols if ld is None else ld
    buf = torch.zeros((rows, ld), dtype=torch.int16)
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return buf.cuda().view(torch.bfloat16)[:, :cols]


def run(tg, A, B, M, N, K, relu=False):
    ld8 = lambda x: max(8, -(-x // 8) * 8)  # noqa: E731
    a = to_dev(A, ld8(K))
    b = to_dev(B, ld8(N))
    cbuf = torch.full((M, ld8(N)), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = tg.tg_gemm_bf16(a.data_ptr(), b.data_ptr(), cbuf.data_ptr(), M, N, K,
                         a.stride(0) if M > 1 else ld8(K), b.stride(0) if K > 1 else ld8(N),
                         cbuf.stride(0) if M > 1 else ld8(N), 1 if relu else 0, s)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_sync_status(s) == tg.TG_OK
    bits = cbuf[:, :N].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return bf16_bits_to_float(bits)


CFGS = ["pair256", "persistent256", "persistent128", "persistent64", "skinny"]
# (64, 4096, 4096): the skinny kernel's four-piece aligned grid in clusters of 4;
# (512, 512, 4096): the pair kernel's last wave in column halves;
# (256, 512, 12288): its tiles in 4 k-pieces
SHAPES = [(1, 1, 1), (7, 7, 7), (129, 127, 1000), (200, 1000, 129), (300, 1000, 1000),
          (64, 2048, 4096), (257, 513, 65), (64, 4096, 4096), (512, 512, 4096),
          (256, 512, 12288)]


@pytest.mark.parametrize("M,N,K", SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SHAPES])
@pytest.mark.parametrize("cfg", CFGS)
def test_bf16_parity_every_kernel(tg, monkeypatch, cfg, M, N, K):
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    A, B = draw_bf16(M, N, K, ("normal", 0, 1), ("normal", 0, 1 / np.sqrt(K)), 500 + M + K)
    for relu in (False, True):
        got = run(tg, A, B, M, N, K, relu)
        want = bf16_bits_to_float(oracle.gemm(A, B, M, N, K, relu=relu, dtype="bf16"))
        check(got, want, K, relu=relu, fmt="bf16", what=f"bf16 {cfg} {M}x{N}x{K}")


def test_bf16_exact_integers(tg):
    """{-1,0,1} inputs, K = 1024: every fp32 partial sum is exact, so the GPU
    rounds the same exact integer to bf16 as the oracle (integers above 256 do
    round): the outputs must be equal."""
    M = N = K = 1024
    A, B = draw_bf16(M, N, K, ("ints", -1, 2), ("ints", -1, 2), 23)
    A[0, :] = bf16_bits(np.ones((1, K)))[0]
    B[:, 0] = bf16_bits(np.ones((K, 1)))[:, 0]  # C[0,0] = 1024, C[0,j] large sums
    for relu in (False, True):
        got = run(tg, A, B, M, N, K, relu)
        want = bf16_bits_to_float(oracle.gemm(A, B, M, N, K, relu=relu, dtype="bf16"))
        check(got, want, K, exact=True, relu=relu, fmt="bf16", what="bf16 ints")
    got = run(tg, A[:100], B, 100, N, K)  # skinny path
    want = bf16_bits_to_float(oracle.gemm(A[:100], B, 100, N, K, dtype="bf16"))
    check(got, want, K, exact=True, fmt="bf16", what="bf16 ints skinny")


@pytest.mark.parametrize("name", ["mlp_8192x28672x4096_relu", "skinny_64x16384x8192"])
def test_bf16_workload_sampled(tg, name):
    w = W.WORKLOADS[name]
    A, B = draw_bf16(w.M, w.N, w.K, w.dist_a, w.dist_b, w.seed)
    a = to_dev(A)
    b = to_dev(B)
    c = tg.gemm(a, b, relu=w.relu)
    tg.sync_status()
    assert c.dtype == torch.bfloat16
    plan = tg.tg_plan_f16(w.M, w.N, w.K, torch.cuda.get_device_properties(0).multi_processor_count)
    rows, cols = W.sample_positions(w.M, w.N, plan.bm if plan.kernel == tg.TG_KERNEL_PERSISTENT
                                    else w.M, plan.bn, w.seed)
    got_bits = c[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    got = bf16_bits_to_float(got_bits.view(torch.int16).cpu().numpy().view(np.uint16))
    want_bits, _ = oracle.gemm_at(A, B, w.K, rows, cols, relu=w.relu, dtype="bf16")
    check(got, bf16_bits_to_float(want_bits), w.K, relu=w.relu, fmt="bf16", what=f"bf16 {name}")


def test_bf16_python_api(tg):
    a = torch.randn(256, 384, device="cuda").to(torch.bfloat16)
    b = (torch.randn(384, 512, device="cuda") * 0.05).to(torch.bfloat16)
    c = tg.gemm(a, b)
    assert c.dtype == torch.bfloat16
    ref = (a.float() @ b.float())
    assert torch.allclose(c.float(), ref, rtol=1e-2, atol=1e-2)
    with pytest.raises(TypeError):
        tg.gemm(a, b.half())
