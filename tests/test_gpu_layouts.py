"""Row-major layouts the tensor memory-access unit cannot address directly
(odd leading dimensions, pointers off a 16-byte boundary): tg_gemm_f16 and
tg_gemm_bf16 stage them through aligned copies and must still match the
oracle, leaving padding untouched."""

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


def placed(bits16: np.ndarray, ld: int, col_off: int, fill: int):
    """A device view of a 16-bit matrix at column offset `col_off` of rows of
    `ld` elements (so the pointer is off 16 B when col_off is not a multiple
    of 8); other elements hold `fill` bits."""
    rows, cols = bits16.shape
    buf = torch.full((rows, ld + col_off), fill, dtype=torch.int16)
    buf[:, col_off:col_off + cols] = torch.from_numpy(np.ascontiguousarray(bits16).view(np.int16))
    full = buf.cuda()
    return full, full[:, col_off:col_off + cols]


LAYOUTS = [
    # (M, N, K, lda, ldb, ldc, a_off, b_off, c_off)
    (7, 7, 7, 7, 7, 7, 0, 0, 0),
    (129, 127, 200, 203, 131, 129, 1, 3, 5),
    (300, 1000, 129, 129, 1001, 1003, 0, 0, 2),
    (64, 1500, 333, 333, 1500, 1500, 2, 0, 0),
    (1000, 200, 64, 64, 201, 200, 0, 1, 0),
    (512, 512, 256, 256, 512, 513, 0, 0, 0),
]
CFGS = ["auto", "pair256", "persistent128", "persistent64", "skinny"]


@pytest.mark.parametrize("layout", LAYOUTS, ids=[f"{l[0]}x{l[1]}x{l[2]}" for l in LAYOUTS])
@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_unaligned_layouts(tg, monkeypatch, layout, cfg, dtype):
    M, N, K, lda, ldb, ldc, ao, bo, co = layout
    if cfg != "auto":
        monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    A64 = W.draw(np.random.default_rng([M + K, 0]), ("normal", 0, 1), M, K)
    B64 = W.draw(np.random.default_rng([M + K, 1]), ("normal", 0, 1 / np.sqrt(K)), K, N)
    if dtype == "bf16":
        conv = lambda x: torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    else:
        conv = lambda x: x.astype(np.float16).view(np.uint16)  # noqa: E731
    A, B = conv(A64), conv(B64)
    sentinel = 0x1234
    fa, a = placed(A, lda, ao, 0x7E00)   # NaN in fp16 padding
    fb, b = placed(B, ldb, bo, 0x7E00)
    fc, c = placed(np.zeros((M, N), np.uint16), ldc, co, sentinel)
    entry = tg.tg_gemm_bf16 if dtype == "bf16" else tg.tg_gemm_f16
    s = torch.cuda.current_stream().cuda_stream
    st = entry(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, fa.stride(0), fb.stride(0),
               fc.stride(0), 1, s)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_sync_status(s) == tg.TG_OK
    got_bits = c.cpu().numpy().view(np.uint16)
    if dtype == "bf16":
        got = bf16_bits_to_float(got_bits)
        want = bf16_bits_to_float(oracle.gemm(A, B, M, N, K, relu=True, dtype="bf16"))
        check(got, want, K, relu=True, fmt="bf16", what=f"bf16 {layout} {cfg}")
    else:
        got = got_bits.view(np.float16)
        check(got, oracle.gemm(A, B, M, N, K, relu=True), K, relu=True, what=f"{layout} {cfg}")
    allc = fc.cpu().numpy().view(np.uint16)
    mask = np.ones_like(allc, dtype=bool)
    mask[:, co:co + N] = False
    assert np.all(allc[mask] == sentinel), "padding of C was written"
