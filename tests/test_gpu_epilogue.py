"""Parity of the extended epilogue (tg_gemm_ex, through the C ABI) against the
oracle's extended GEMM on a GB300:

    C = out( act( A·B + bias ) + R )

on every kernel (forced with TGEMM_FORCE_CFG), for fp16 and bf16 inputs,
16-bit and fp32 outputs, with and without bias / residual / ReLU; K == 0;
a residual that is C itself; layouts that need staging or scalar loads; and
sampled outputs at the MLP layer's full size.

Tolerances.  16-bit output: the rule of parity.py (2 ulp of the output type
at the oracle value + 1e-3·sqrt(K)); the kernel's two extra fp32 additions
(bias, residual) each add at most half an fp32 ulp, far inside it.  fp32
output: the oracle is the exact value rounded once to fp32; the kernel
accumulates K products in fp32 and then adds bias and R in fp32, each step
erring by at most 2^-23 of the running magnitude, bounded by
T = sum_k |a_ik b_kj| + |bias_j| + |R_ij|.  So
    |gpu - oracle| <= 2 ulp32(oracle) + (K + 2) * 2^-23 * T.
On integer inputs ({-1, 0, 1} operands, K <= 2048, integer bias and
residual) every intermediate is an integer below 2^24, exact in fp32, so the
fp32 output must equal the oracle bit for bit.
"""

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


CFGS = ["pair256", "persistent256", "persistent128", "persistent64", "skinny"]
TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


def bits16(x64: np.ndarray, fmt: str) -> np.ndarray:
    """float64 values rounded to the 16-bit type by torch, as uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x64)).to(TDT[fmt])
    return t.view(torch.int16).numpy().view(np.uint16)


def decode(bits: np.ndarray, fmt: str) -> np.ndarray:
    if fmt == "bf16":
        return bf16_bits_to_float(bits)
    return np.ascontiguousarray(bits).view(np.float16).astype(np.float64)


def dev16(bits: np.ndarray, fmt: str, ld: int | None = None, offset: int = 0):
    """A device view of a 16-bit matrix with row stride ld, starting `offset`
    elements into its buffer (offset 1 gives a pointer that is not 16-byte
    aligned)."""
    rows, cols = bits.shape
    ld = cols if ld is None else ld
    buf = torch.zeros(rows * ld + offset + 8, dtype=torch.int16)
    view = buf[offset:offset + rows * ld].view(rows, ld)
    view[:, :cols] = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return buf.cuda().view(TDT[fmt])[offset:offset + rows * ld].view(rows, ld)[:, :cols]


def out_buffer(M, N, out, fmt, ld=None, offset=0):
    ld = N if ld is None else ld
    dt = torch.float32 if out == "f32" else TDT[fmt]
    buf = torch.full((M * ld + offset + 8,), float("nan"), dtype=dt, device="cuda")
    return buf[offset:offset + M * ld].view(M, ld)[:, :N]


def abs_scale(A64, B64, bias, R64):
    """T = sum_k |a_ik b_kj| + |bias_j| + |R_ij| in float64."""
    T = np.abs(A64) @ np.abs(B64)
    if bias is not None:
        T = T + np.abs(bias.astype(np.float64))[None, :]
    if R64 is not None:
        T = T + np.abs(R64)
    return T


def ulp32(x):
    a = np.abs(np.asarray(x, dtype=np.float64))
    out = np.full(a.shape, 2.0 ** -149)
    nz = a >= 2.0 ** -126
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    out[nz] = np.exp2(e[nz] - 23.0)
    return out


def check_f32(got, want, K, T, *, exact=False, what=""):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(want, dtype=np.float32).astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    if exact:
        bad = g != r
        assert not np.any(bad), f"{what}: {int(bad.sum())} differ, first {np.argwhere(bad)[:5]}"
        return
    tol = 2.0 * ulp32(r) + (K + 2) * 2.0 ** -23 * T
    err = np.abs(g - r)
    bad = err > tol
    assert not np.any(bad), (f"{what}: {int(bad.sum())} of {g.size} outside tolerance; worst "
                             f"{err.max():.3g} vs tol {tol.flat[np.argmax(err - tol)]:.3g}")


def call_ex(tg, fmt, a, b, c, M, N, K, *, relu=False, bias=None, resid=None, out="f16",
            lda=None, ldb=None, ldc=None, ldr=None):
    ld = lambda t, cols: (t.stride(0) if t.shape[0] > 1 else max(8, -(-cols // 8) * 8))  # noqa
    in_code = tg.TG_DTYPE_BF16 if fmt == "bf16" else tg.TG_DTYPE_F16
    out_code = tg.TG_DTYPE_F32 if out == "f32" else in_code
    epi = tg.tg_epilogue_ex_t(1 if relu else 0, out_code,
                              bias.data_ptr() if bias is not None else None,
                              resid.data_ptr() if resid is not None else None,
                              (ldr if ldr is not None else ld(resid, N)) if resid is not None else 0)
    s = torch.cuda.current_stream().cuda_stream
    st = tg.tg_gemm_ex(in_code, a.data_ptr() if a is not None else None,
                       b.data_ptr() if b is not None else None, c.data_ptr(), M, N, K,
                       lda if lda is not None else (ld(a, K) if a is not None else K),
                       ldb if ldb is not None else (ld(b, N) if b is not None else N),
                       ldc if ldc is not None else ld(c, N), epi, s)
    return st


def host_out(c, out, fmt):
    if out == "f32":
        return c.float().cpu().numpy().astype(np.float64)
    bits = c.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return decode(bits, fmt)


def draw_case(M, N, K, fmt, seed, *, integer=False):
    rng = lambda i: np.random.default_rng([seed, i])  # noqa: E731
    if integer:
        A64 = W.draw(rng(0), ("ints", -1, 2), M, K)
        B64 = W.draw(rng(1), ("ints", -1, 2), K, N)
        bias = rng(2).integers(-8, 9, size=N).astype(np.float32)
        R64 = rng(3).integers(-64, 65, size=(M, N)).astype(np.float64)
    else:
        A64 = W.draw(rng(0), ("normal", 0, 1), M, K)
        B64 = W.draw(rng(1), ("normal", 0, 1 / np.sqrt(max(K, 1))), K, N)
        bias = rng(2).normal(0.0, 0.5, size=N).astype(np.float32)
        R64 = rng(3).normal(0.0, 1.0, size=(M, N))
    A, B, R = bits16(A64, fmt), bits16(B64, fmt), bits16(R64, fmt)
    return A, B, bias, R, decode(A, fmt), decode(B, fmt), decode(R, fmt)


VARIANTS = [  # (relu, bias, residual, out)
    (False, True, False, "same"),
    (True, True, True, "same"),
    (False, False, True, "same"),
    (False, False, False, "f32"),
    (True, True, True, "f32"),
]
# 512×512×4096 and 300×700×2048: the pair kernel runs its tail tiles as
# column halves (256×128 products); 64×4096×4096: the skinny kernel's aligned
# grid (32 tiles in 4 equal k pieces).  The pair kernel's k-pieces, whose
# epilogue runs on summed fp32 partials, are test_epilogue_pair_k_pieces.
SHAPES = [(1, 1, 1), (129, 127, 1000), (300, 1000, 129), (64, 2048, 520), (257, 513, 65),
          (512, 512, 4096), (300, 700, 2048), (64, 4096, 4096)]


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SHAPES])
@pytest.mark.parametrize("cfg", CFGS)
def test_epilogue_every_kernel(tg, monkeypatch, cfg, M, N, K, fmt):
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    A, B, bias, R, A64, B64, R64 = draw_case(M, N, K, fmt, 700 + M + N + K)
    a, b = dev16(A, fmt), dev16(B, fmt)
    bias_d = torch.from_numpy(bias).cuda()
    r_d = dev16(R, fmt)
    for relu, use_bias, use_r, out in VARIANTS:
        out_t = "f32" if out == "f32" else fmt
        c = out_buffer(M, N, out_t, fmt)
        st = call_ex(tg, fmt, a, b, c, M, N, K, relu=relu, bias=bias_d if use_bias else None,
                     resid=r_d if use_r else None, out=out_t)
        assert st == tg.TG_OK, tg.tg_status_string(st)
        assert tg.tg_sync_status(torch.cuda.current_stream().cuda_stream) == tg.TG_OK
        got = host_out(c, out_t, fmt)
        want = oracle.gemm_ex(A, B, M, N, K, relu=relu, bias=bias if use_bias else None,
                              R=R if use_r else None, in_dtype=fmt, out_dtype=out_t)
        what = f"{cfg} {fmt} {M}x{N}x{K} relu={relu} bias={use_bias} R={use_r} out={out_t}"
        if out_t == "f32":
            T = abs_scale(A64, B64, bias if use_bias else None, R64 if use_r else None)
            check_f32(got, want, K, T, what=what)
        else:
            check(got, decode(want, fmt) if fmt == "bf16" else want, K,
                  relu=relu and not use_r, fmt=fmt, what=what)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_epilogue_pair_k_pieces(tg, monkeypatch, fmt):
    """256×512×12288 on the pair kernel: 2 tiles, each cut into 4 k-pieces;
    the last piece in applies every epilogue variant to the summed partials."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", "pair256")
    M, N, K = 256, 512, 12288
    A, B, bias, R, A64, B64, R64 = draw_case(M, N, K, fmt, 4321)
    a, b = dev16(A, fmt), dev16(B, fmt)
    bias_d = torch.from_numpy(bias).cuda()
    r_d = dev16(R, fmt)
    for relu, use_bias, use_r, out in VARIANTS:
        out_t = "f32" if out == "f32" else fmt
        c = out_buffer(M, N, out_t, fmt)
        st = call_ex(tg, fmt, a, b, c, M, N, K, relu=relu, bias=bias_d if use_bias else None,
                     resid=r_d if use_r else None, out=out_t)
        assert st == tg.TG_OK, tg.tg_status_string(st)
        assert tg.tg_sync_status(torch.cuda.current_stream().cuda_stream) == tg.TG_OK
        launched = tg.tg_debug_last_launch()
        if launched.grid == 16:  # all pairs resident: the planned cut
            assert launched.split_k == 4 and launched.split_n == 1
        got = host_out(c, out_t, fmt)
        want = oracle.gemm_ex(A, B, M, N, K, relu=relu, bias=bias if use_bias else None,
                              R=R if use_r else None, in_dtype=fmt, out_dtype=out_t)
        what = f"pair k-pieces {fmt} relu={relu} bias={use_bias} R={use_r} out={out_t}"
        if out_t == "f32":
            T = abs_scale(A64, B64, bias if use_bias else None, R64 if use_r else None)
            check_f32(got, want, K, T, what=what)
        else:
            check(got, decode(want, fmt) if fmt == "bf16" else want, K,
                  relu=relu and not use_r, fmt=fmt, what=what)


@pytest.mark.parametrize("cfg", ["pair256", "persistent128", "persistent64", "skinny"])
def test_plain_and_full_builds_interleaved(tg, monkeypatch, cfg):
    """Plain epilogues (ReLU or none, 16-bit out) run a build of each kernel
    with the other epilogue paths compiled out.  Calls of both builds queued
    back to back on one stream (dependent launch between different kernels),
    with one synchronisation at the end, each match the oracle.  The skinny
    case (96×640×4096) splits every tile into k-pieces, so both builds' fix-up
    paths run."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    M, N, K, fmt = (96, 640, 4096, "f16") if cfg == "skinny" else (384, 640, 512, "f16")
    A, B, bias, R, A64, B64, R64 = draw_case(M, N, K, fmt, 97)
    a, b = dev16(A, fmt), dev16(B, fmt)
    bias_d = torch.from_numpy(bias).cuda()
    r_d = dev16(R, fmt)
    plan = [(True, False, False, fmt), (False, True, True, fmt), (False, False, False, "f32"),
            (False, False, False, fmt), (True, True, False, "f32"), (True, False, False, fmt)]
    outs = []
    for relu, use_bias, use_r, out_t in plan:
        c = out_buffer(M, N, out_t, fmt)
        st = call_ex(tg, fmt, a, b, c, M, N, K, relu=relu, bias=bias_d if use_bias else None,
                     resid=r_d if use_r else None, out=out_t)
        assert st == tg.TG_OK, tg.tg_status_string(st)
        outs.append(c)
    assert tg.tg_sync_status(torch.cuda.current_stream().cuda_stream) == tg.TG_OK
    for (relu, use_bias, use_r, out_t), c in zip(plan, outs):
        got = host_out(c, out_t, fmt)
        want = oracle.gemm_ex(A, B, M, N, K, relu=relu, bias=bias if use_bias else None,
                              R=R if use_r else None, in_dtype=fmt, out_dtype=out_t)
        what = f"{cfg} interleaved relu={relu} bias={use_bias} R={use_r} out={out_t}"
        if out_t == "f32":
            T = abs_scale(A64, B64, bias if use_bias else None, R64 if use_r else None)
            check_f32(got, want, K, T, what=what)
        else:
            check(got, want, K, relu=relu and not use_r, fmt=fmt, what=what)


@pytest.mark.parametrize("cfg", CFGS)
def test_epilogue_exact_integers_f32(tg, monkeypatch, cfg):
    """Integer operands, bias and residual: the fp32 output is exact, so it
    must match the oracle bit for bit (this pins the fp32 store layout)."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    M, N, K = (100, 520, 1024) if cfg == "skinny" else (300, 520, 1024)
    for fmt in ("f16", "bf16"):
        A, B, bias, R, *_ = draw_case(M, N, K, fmt, 31, integer=True)
        a, b, r_d = dev16(A, fmt), dev16(B, fmt), dev16(R, fmt)
        bias_d = torch.from_numpy(bias).cuda()
        for relu in (False, True):
            c = out_buffer(M, N, "f32", fmt)
            st = call_ex(tg, fmt, a, b, c, M, N, K, relu=relu, bias=bias_d, resid=r_d, out="f32")
            assert st == tg.TG_OK
            got = host_out(c, "f32", fmt)
            want = oracle.gemm_ex(A, B, M, N, K, relu=relu, bias=bias, R=R, in_dtype=fmt,
                                  out_dtype="f32")
            check_f32(got, want, K, None, exact=True, what=f"{cfg} {fmt} relu={relu}")


@pytest.mark.parametrize("out", ["same", "f32"])
def test_epilogue_k0(tg, out):
    """K == 0: C = out(act(bias) + R); A and B may be NULL."""
    M, N, fmt = 37, 91, "f16"
    _, _, bias, R, *_ = draw_case(M, N, 1, fmt, 5)
    bias_d, r_d = torch.from_numpy(bias).cuda(), dev16(R, fmt)
    out_t = "f32" if out == "f32" else fmt
    for relu in (False, True):
        c = out_buffer(M, N, out_t, fmt)
        st = call_ex(tg, fmt, None, None, c, M, N, 0, relu=relu, bias=bias_d, resid=r_d,
                     out=out_t)
        assert st == tg.TG_OK
        torch.cuda.synchronize()
        got = host_out(c, out_t, fmt)
        want = oracle.gemm_ex(np.zeros((M, 1), np.uint16), np.zeros((1, N), np.uint16), M, N, 0,
                              relu=relu, bias=bias, R=R, in_dtype=fmt, out_dtype=out_t)
        want = np.asarray(want, dtype=np.float64)
        assert np.array_equal(got, want), f"K=0 relu={relu} out={out_t}"


@pytest.mark.parametrize("cfg", CFGS)
def test_residual_is_output(tg, monkeypatch, cfg):
    """R == C (same buffer, ldr == ldc): every element is read before it is
    overwritten, so the in-place update equals the out-of-place one."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    M = 96 if cfg == "skinny" else 333
    N, K, fmt = 777, 300, "f16"
    A, B, bias, R, *_ = draw_case(M, N, K, fmt, 77)
    a, b = dev16(A, fmt), dev16(B, fmt)
    bias_d = torch.from_numpy(bias).cuda()
    c = dev16(R, fmt, ld=784)
    st = call_ex(tg, fmt, a, b, c, M, N, K, relu=True, bias=bias_d, resid=c, out=fmt)
    assert st == tg.TG_OK
    got = host_out(c, fmt, fmt)
    want = oracle.gemm_ex(A, B, M, N, K, relu=True, bias=bias, R=R, in_dtype="f16",
                          out_dtype="f16")
    check(got, want, K, what=f"in-place {cfg}")


@pytest.mark.parametrize("cfg", CFGS)
def test_epilogue_unaligned_layouts(tg, monkeypatch, cfg):
    """fp32 C with an odd ldc and an unaligned pointer (computed in staging and
    copied back); residual with an odd ldr and an unaligned pointer; bias at a
    4-byte (not 16-byte) offset: the scalar load paths."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    M, N, K, fmt = (120 if cfg == "skinny" else 260), 203, 150, "bf16"
    A, B, bias, R, A64, B64, R64 = draw_case(M, N, K, fmt, 9)
    a, b = dev16(A, fmt, ld=157, offset=1), dev16(B, fmt, ld=211, offset=3)
    r_d = dev16(R, fmt, ld=205, offset=1)
    bias_buf = torch.zeros(N + 1, dtype=torch.float32, device="cuda")
    bias_buf[1:] = torch.from_numpy(bias).cuda()
    bias_d = bias_buf[1:]
    for out in ("f32", fmt):
        c = out_buffer(M, N, out, fmt, ld=N + 2, offset=1)
        st = call_ex(tg, fmt, a, b, c, M, N, K, relu=False, bias=bias_d, resid=r_d, out=out)
        assert st == tg.TG_OK, tg.tg_status_string(st)
        got = host_out(c, out, fmt)
        want = oracle.gemm_ex(A, B, M, N, K, bias=bias, R=R, in_dtype=fmt, out_dtype=out)
        if out == "f32":
            check_f32(got, want, K, abs_scale(A64, B64, bias, R64), what=f"{cfg} f32 staged")
        else:
            check(got, decode(want, fmt), K, fmt=fmt, what=f"{cfg} bf16 unaligned")


def test_python_api_epilogue(tg):
    """tiled_fp16_gemm_gb300.gemm(..., bias=, residual=, out_dtype=)."""
    M, N, K, fmt = 200, 300, 400, "f16"
    A, B, bias, R, A64, B64, R64 = draw_case(M, N, K, fmt, 3)
    a, b, r = dev16(A, fmt), dev16(B, fmt), dev16(R, fmt)
    bias_d = torch.from_numpy(bias).cuda()
    c = tg.gemm(a, b, relu=True, bias=bias_d, residual=r, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert c.dtype == torch.float32 and tuple(c.shape) == (M, N)
    want = oracle.gemm_ex(A, B, M, N, K, relu=True, bias=bias, R=R, out_dtype="f32")
    check_f32(c.cpu().numpy(), want, K, abs_scale(A64, B64, bias, R64), what="api f32")
    c16 = tg.gemm(a, b, bias=bias_d)
    torch.cuda.synchronize()
    want16 = oracle.gemm_ex(A, B, M, N, K, bias=bias)
    check(c16.cpu().numpy(), want16, K, what="api bias")
    with pytest.raises(TypeError):
        tg.gemm(a, b, out_dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        tg.gemm(a, b, bias=bias_d[:-1])
    with pytest.raises(ValueError):
        tg.gemm(a, b, residual=r[:, :-1])


def test_epilogue_mlp_full_size_sampled(tg):
    """8192×28672×4096 (the MLP layer) with bias, ReLU and residual, fp32 and
    fp16 outputs, through the planner's kernel: sampled outputs against the
    oracle computed one by one."""
    M, N, K = 8192, 28672, 4096
    fmt = "f16"
    A, B = (x.view(np.uint16) for x in W.workload_inputs(W.WORKLOADS["mlp_8192x28672x4096_relu"]))
    rng = np.random.default_rng(11)
    bias = rng.normal(0.0, 0.5, size=N).astype(np.float32)
    R = bits16(rng.normal(0.0, 1.0, size=(M, N)), fmt)
    a, b, r_d = dev16(A, fmt), dev16(B, fmt), dev16(R, fmt)
    bias_d = torch.from_numpy(bias).cuda()
    rows, cols = W.sample_positions(M, N, 256, 256, seed=12)
    absA = np.abs(A.view(np.float16).astype(np.float32))
    absB = np.abs(B.view(np.float16).astype(np.float32))
    T = np.empty(rows.size, dtype=np.float64)
    for i in range(0, rows.size, 8192):  # sum_k |a_ik b_kj| at the sampled positions
        r, c = rows[i:i + 8192], cols[i:i + 8192]
        T[i:i + 8192] = np.einsum("ik,ki->i", absA[r], absB[:, c], dtype=np.float64)
    T += np.abs(bias[cols]) + np.abs(decode(R[rows, cols], fmt))
    for out in ("f32", fmt):
        c = out_buffer(M, N, out, fmt)
        st = call_ex(tg, fmt, a, b, c, M, N, K, relu=True, bias=bias_d, resid=r_d, out=out)
        assert st == tg.TG_OK
        assert tg.tg_sync_status(torch.cuda.current_stream().cuda_stream) == tg.TG_OK
        got_all = c[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
        got = host_out(got_all.view(1, -1), out, fmt).ravel()
        want, _ = oracle.gemm_ex_at(A, B, K, rows, cols, relu=True, bias=bias, R=R,
                                    in_dtype=fmt, out_dtype=out)
        if out == "f32":
            check_f32(got, want, K, T, what="mlp f32 sampled")
        else:
            check(got, want, K, what="mlp f16 sampled")
        del c
