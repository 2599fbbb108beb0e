"""Python binding for libtgemm (dense FP16 GEMM on GB300, sm_103a).

Argument marshalling only: every step of C = epi(A·B) runs in the CUDA
kernels of ``libtgemm.so``, called through its C ABI (``include/tgemm.h``).
PyTorch is used for device memory and streams.  There is no fallback: if the
shared library is missing, the first call raises ImportError.

Build the library with ``tiled_fp16_gemm_gb300.build.build()`` (nvcc, sm_103a).
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtgemm.so")

TG_EPI_NONE = 0
TG_EPI_RELU = 1

TG_OK = 0
TG_ERR_INVALID_VALUE = 1
TG_ERR_MISALIGNED = 2
TG_ERR_UNSUPPORTED_DEVICE = 3
TG_ERR_LAUNCH = 4
TG_ERR_NO_MEMORY = 5
TG_ERR_TIMEOUT = 6

TG_DTYPE_F16 = 0
TG_DTYPE_BF16 = 1
TG_DTYPE_F32 = 2

TG_KERNEL_NONE = 0
TG_KERNEL_FILL = 1
TG_KERNEL_PERSISTENT = 2
TG_KERNEL_SKINNY = 3

#: every symbol include/tgemm.h declares
EXPORTS = (
    "tg_gemm_f16", "tg_sync_status", "tg_status_string", "tg_version", "tg_plan_f16",
    "tg_tile_coord", "tg_ring_bytes", "tg_debug_set_wait_timeout_ns", "tg_debug_inject",
    "tg_gemm_f16_noalloc", "tg_gemm_bf16", "tg_gemm_ex", "tg_gemm_mxfp4", "tg_gemm_sp24",
    "tg_gemm_f16_host", "tg_plan_f16_limits", "tg_device_limits", "tg_debug_last_launch",
    "tg_debug_map_cache_stats",
)

#: bytes of the library's fixed scratch array used by tg_gemm_f16_noalloc
TG_NOALLOC_SCRATCH_BYTES = 24 * 1024 * 1024


class tg_plan_t(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int32), ("bm", ctypes.c_int32), ("bn", ctypes.c_int32),
        ("bk", ctypes.c_int32), ("stages", ctypes.c_int32), ("mma_m", ctypes.c_int32),
        ("mma_n", ctypes.c_int32), ("tiles_m", ctypes.c_int64), ("tiles_n", ctypes.c_int64),
        ("k_blocks", ctypes.c_int64), ("num_tiles", ctypes.c_int64), ("grid", ctypes.c_int64),
        ("threads", ctypes.c_int32), ("group_m", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int64), ("ring_bytes", ctypes.c_int64),
        ("split_k", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
        ("cluster", ctypes.c_int32), ("split_n", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class tg_epilogue_ex_t(ctypes.Structure):
    _fields_ = [
        ("activation", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
        ("bias", ctypes.c_void_p), ("residual", ctypes.c_void_p), ("ldr", ctypes.c_int64),
    ]


_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_lib = None


def _L():
    """Load libtgemm.so on first use; there is no fallback if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libtgemm.so not found at {LIB_PATH}; build it with "
            "`python -m tiled_fp16_gemm_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    lib.tg_gemm_f16.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
                                _vp]
    lib.tg_gemm_f16.restype = ctypes.c_int
    lib.tg_gemm_bf16.argtypes = lib.tg_gemm_f16.argtypes
    lib.tg_gemm_bf16.restype = ctypes.c_int
    lib.tg_gemm_f16_host.argtypes = lib.tg_gemm_f16.argtypes
    lib.tg_gemm_f16_host.restype = ctypes.c_int
    lib.tg_gemm_ex.argtypes = [ctypes.c_int32, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64,
                               ctypes.POINTER(tg_epilogue_ex_t), _vp]
    lib.tg_gemm_ex.restype = ctypes.c_int
    lib.tg_gemm_mxfp4.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, _i64,
                                  ctypes.POINTER(tg_epilogue_ex_t), _vp]
    lib.tg_gemm_mxfp4.restype = ctypes.c_int
    lib.tg_gemm_sp24.argtypes = [ctypes.c_int32, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                 _i64, _i64, _i64, ctypes.POINTER(tg_epilogue_ex_t), _vp]
    lib.tg_gemm_sp24.restype = ctypes.c_int
    lib.tg_sync_status.argtypes = [_vp]
    lib.tg_sync_status.restype = ctypes.c_int
    lib.tg_status_string.argtypes = [ctypes.c_int]
    lib.tg_status_string.restype = ctypes.c_char_p
    lib.tg_version.restype = ctypes.c_char_p
    lib.tg_plan_f16.argtypes = [_i64, _i64, _i64, ctypes.c_int32, ctypes.POINTER(tg_plan_t)]
    lib.tg_plan_f16.restype = ctypes.c_int
    lib.tg_tile_coord.argtypes = [ctypes.POINTER(tg_plan_t), _i64, ctypes.POINTER(_i64),
                                  ctypes.POINTER(_i64)]
    lib.tg_tile_coord.restype = ctypes.c_int
    lib.tg_ring_bytes.argtypes = [ctypes.c_int32] * 5
    lib.tg_ring_bytes.restype = _i64
    lib.tg_debug_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.tg_debug_set_wait_timeout_ns.restype = None
    lib.tg_debug_inject.argtypes = [ctypes.c_int32]
    lib.tg_debug_inject.restype = None
    lib.tg_plan_f16_limits.argtypes = [_i64, _i64, _i64] + [ctypes.c_int32] * 4 + [
        ctypes.POINTER(tg_plan_t)]
    lib.tg_plan_f16_limits.restype = ctypes.c_int
    lib.tg_device_limits.argtypes = [ctypes.POINTER(ctypes.c_int32)] * 4
    lib.tg_device_limits.restype = ctypes.c_int
    lib.tg_debug_last_launch.argtypes = [ctypes.POINTER(tg_plan_t)]
    lib.tg_debug_last_launch.restype = ctypes.c_int
    lib.tg_debug_map_cache_stats.argtypes = [ctypes.POINTER(ctypes.c_uint64)] * 2
    lib.tg_debug_map_cache_stats.restype = None
    _lib = lib
    return lib


def library():
    """The loaded ctypes.CDLL of libtgemm.so."""
    return _L()


class TgemmError(RuntimeError):
    def __init__(self, status: int, what: str = "tg_gemm_f16"):
        self.status = status
        super().__init__(f"{what}: {tg_status_string(status)}")


# ------------------------------------------------------------------ raw C ABI

def tg_gemm_f16(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                epilogue: int, stream: int | None) -> int:
    """The C entry point with integer device pointers; returns the status code."""
    return _L().tg_gemm_f16(A, B, C, M, N, K, lda, ldb, ldc, epilogue, stream or None)


def tg_gemm_bf16(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                 epilogue: int, stream: int | None) -> int:
    """The bfloat16 entry point with integer device pointers; returns the status code."""
    return _L().tg_gemm_bf16(A, B, C, M, N, K, lda, ldb, ldc, epilogue, stream or None)


def tg_gemm_f16_host(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                     ldc: int, epilogue: int, stream: int | None) -> int:
    """The C entry point with integer HOST pointers; returns the status code."""
    return _L().tg_gemm_f16_host(A, B, C, M, N, K, lda, ldb, ldc, epilogue, stream or None)


def tg_gemm_ex(in_dtype: int, A: int, B: int, C: int, M: int, N: int, K: int, lda: int,
               ldb: int, ldc: int, epi: tg_epilogue_ex_t | None, stream: int | None) -> int:
    """C = out(act(A·B + bias) + R) with integer device pointers; returns the status code."""
    return _L().tg_gemm_ex(in_dtype, A, B, C, M, N, K, lda, ldb, ldc,
                           ctypes.byref(epi) if epi is not None else None, stream or None)


def tg_gemm_mxfp4(A: int, Bq: int, Bscale: int, C: int, M: int, N: int, K: int, lda: int,
                  ldbq: int, ldbs: int, ldc: int, epi: tg_epilogue_ex_t | None,
                  stream: int | None) -> int:
    """C = out(act(A·Bdeq + bias) + R) with B in MXFP4 (packed E2M1 codes and
    E8M0 scales per 32 k), integer device pointers; returns the status code."""
    return _L().tg_gemm_mxfp4(A, Bq, Bscale, C, M, N, K, lda, ldbq, ldbs, ldc,
                              ctypes.byref(epi) if epi is not None else None, stream or None)


def tg_gemm_sp24(in_dtype: int, Ac: int, E: int, B: int, C: int, M: int, N: int, K: int,
                 ldac: int, lde: int, ldb: int, ldc: int, epi: tg_epilogue_ex_t | None,
                 stream: int | None) -> int:
    """C = out(act(A·B + bias) + R) with A 2:4 sparse (compressed values Ac and
    metadata words E), integer device pointers; returns the status code."""
    return _L().tg_gemm_sp24(in_dtype, Ac, E, B, C, M, N, K, ldac, lde, ldb, ldc,
                             ctypes.byref(epi) if epi is not None else None, stream or None)


def tg_sync_status(stream: int | None) -> int:
    return _L().tg_sync_status(stream or None)


def tg_status_string(status: int) -> str:
    return _L().tg_status_string(status).decode()


def tg_version() -> str:
    return _L().tg_version().decode()


def tg_plan_f16(M: int, N: int, K: int, num_sms: int) -> tg_plan_t:
    plan = tg_plan_t()
    st = _L().tg_plan_f16(M, N, K, num_sms, ctypes.byref(plan))
    if st != TG_OK:
        raise TgemmError(st, "tg_plan_f16")
    return plan


def tg_plan_f16_limits(M: int, N: int, K: int, num_sms: int, max_pairs: int,
                       max_quads_narrow: int, max_quads_wide: int) -> tg_plan_t:
    plan = tg_plan_t()
    st = _L().tg_plan_f16_limits(M, N, K, num_sms, max_pairs, max_quads_narrow, max_quads_wide,
                                 ctypes.byref(plan))
    if st != TG_OK:
        raise TgemmError(st, "tg_plan_f16_limits")
    return plan


def tg_device_limits() -> tuple[int, int, int, int]:
    """(num_sms, max_pairs, max_quads_narrow, max_quads_wide) of the current device."""
    v = [ctypes.c_int32() for _ in range(4)]
    st = _L().tg_device_limits(*[ctypes.byref(x) for x in v])
    if st != TG_OK:
        raise TgemmError(st, "tg_device_limits")
    return tuple(x.value for x in v)


def tg_debug_last_launch() -> tg_plan_t:
    plan = tg_plan_t()
    st = _L().tg_debug_last_launch(ctypes.byref(plan))
    if st != TG_OK:
        raise TgemmError(st, "tg_debug_last_launch")
    return plan


def tg_debug_map_cache_stats() -> tuple[int, int]:
    """(hits, misses) of the library's tensor-map cache since it was loaded."""
    h, m = ctypes.c_uint64(), ctypes.c_uint64()
    _L().tg_debug_map_cache_stats(ctypes.byref(h), ctypes.byref(m))
    return h.value, m.value


def tg_tile_coord(plan: tg_plan_t, tile: int) -> tuple[int, int]:
    m, n = _i64(), _i64()
    st = _L().tg_tile_coord(ctypes.byref(plan), tile, ctypes.byref(m), ctypes.byref(n))
    if st != TG_OK:
        raise TgemmError(st, "tg_tile_coord")
    return m.value, n.value


def tg_ring_bytes(bm: int, bn: int, bk: int, stages: int, elem_bytes: int) -> int:
    return _L().tg_ring_bytes(bm, bn, bk, stages, elem_bytes)


def tg_debug_set_wait_timeout_ns(ns: int) -> None:
    _L().tg_debug_set_wait_timeout_ns(ns)


def tg_debug_inject(mode: int) -> None:
    _L().tg_debug_inject(mode)


def tg_gemm_f16_noalloc(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                        ldc: int, epilogue: int, stream: int | None) -> int:
    """C = epi(A·B) for M <= 128 with no device allocation: the split-K
    scratch lives in a fixed 24 MiB array inside the library.  For callers
    that cannot allocate device memory at call time.  Calls that overlap on
    the GPU share that array and race; the first call on a device does a
    one-time set-up and should come before any stream capture.  Returns the
    status code."""
    lib = _L()
    fn = lib.tg_gemm_f16_noalloc
    fn.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _vp]
    fn.restype = ctypes.c_int
    return fn(A, B, C, M, N, K, lda, ldb, ldc, epilogue, stream or None)


# ------------------------------------------------------------------ torch helpers

def _check_operand(t, name: str):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError(f"{name} must be float16 or bfloat16, got {t.dtype}")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major (unit column stride)")


def _ld(t) -> int:
    if t.shape[0] > 1:
        return int(t.stride(0))
    # a single row: the row stride is never used, pass the 8-aligned width
    return max(8, (int(t.shape[1]) + 7) // 8 * 8)


def gemm(a, b, relu: bool = False, out=None, stream=None, *, bias=None, residual=None,
         out_dtype=None):
    """C = out(act(a @ b + bias) + residual) for CUDA float16 (or bfloat16)
    tensors a (M×K) and b (K×N); act = ReLU if ``relu`` else identity.

    bias: optional float32 tensor of N elements (added to the fp32
    accumulator before the activation).  residual: optional M×N tensor of a's
    dtype (added after the activation; may be ``out`` itself).  out_dtype:
    a's dtype (default) or torch.float32.  Any row-major 2-D views are
    accepted (unit column stride); ``out`` (M×N) is written in place when
    given.  Runs on ``stream`` (default: torch's current stream of a's device).
    """
    import torch
    _check_operand(a, "a")
    _check_operand(b, "b")
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if not (a.is_cuda and b.is_cuda and a.device == b.device):
        raise ValueError("a and b must be CUDA tensors on the same device")
    if a.dtype != b.dtype:
        raise TypeError(f"a and b must share a dtype, got {a.dtype} and {b.dtype}")
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else a.dtype
    if out_dtype not in (a.dtype, torch.float32):
        raise TypeError(f"out_dtype must be {a.dtype} or torch.float32, got {out_dtype}")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    else:
        if out.dtype != out_dtype or out.dim() != 2 or tuple(out.shape) != (M, N) \
                or out.device != a.device:
            raise ValueError("out must be M×N on a's device with dtype out_dtype")
        if N > 1 and out.stride(1) != 1:
            raise ValueError("out must be row-major (unit column stride)")
    extended = bias is not None or residual is not None or out_dtype == torch.float32
    if bias is not None:
        if not isinstance(bias, torch.Tensor) or bias.dtype != torch.float32 \
                or bias.device != a.device or bias.numel() != N or bias.dim() != 1 \
                or (N > 1 and bias.stride(0) != 1):
            raise ValueError("bias must be a contiguous float32 CUDA tensor of N elements")
    if residual is not None:
        _check_operand(residual, "residual")
        if residual.dtype != a.dtype or tuple(residual.shape) != (M, N) \
                or residual.device != a.device:
            raise ValueError("residual must be M×N on a's device with a's dtype")
    in_code = TG_DTYPE_BF16 if a.dtype == torch.bfloat16 else TG_DTYPE_F16
    with torch.cuda.device(a.device):
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        if extended:
            epi = tg_epilogue_ex_t(
                TG_EPI_RELU if relu else TG_EPI_NONE,
                TG_DTYPE_F32 if out_dtype == torch.float32 else in_code,
                bias.data_ptr() if bias is not None else None,
                residual.data_ptr() if residual is not None else None,
                _ld(residual) if residual is not None else 0)
            st = tg_gemm_ex(in_code, a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K,
                            _ld(a), _ld(b), _ld(out), epi, s.cuda_stream)
            what = "tg_gemm_ex"
        else:
            entry = tg_gemm_bf16 if in_code == TG_DTYPE_BF16 else tg_gemm_f16
            st = entry(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, _ld(a), _ld(b),
                       _ld(out), TG_EPI_RELU if relu else TG_EPI_NONE, s.cuda_stream)
            what = entry.__name__
    if st != TG_OK:
        raise TgemmError(st, what)
    return out


def gemm_mxfp4(a, bq, bscale, N: int, relu: bool = False, out=None, stream=None, *, bias=None,
               residual=None, out_dtype=None):
    """C = out(act(a @ Bdeq + bias) + residual) with the weight in MXFP4.

    a: CUDA float16 tensor M×K (row-major).  bq: CUDA uint8 tensor of N rows
    (one per weight column, the [out][in] orientation) of packed E2M1 codes
    along k, low nibble first (row stride a multiple of 16 bytes, at least
    ceil(K/2)); bscale: CUDA uint8 tensor of ceil(K/32) rows of E8M0 scales
    (row stride a multiple of 16, at least N).  N is the number of weight
    columns.  bias, residual, out_dtype, out and stream as for ``gemm``.
    """
    import torch
    _check_operand(a, "a")
    if a.dtype != torch.float16:
        raise TypeError("a must be float16 for the MXFP4 GEMM")
    M, K = a.shape
    for t, name, rows, width in ((bq, "bq", N, (K + 1) // 2), (bscale, "bscale", (K + 31) // 32, N)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or t.dim() != 2:
            raise TypeError(f"{name} must be a 2-D uint8 tensor")
        if t.shape[0] != rows or t.shape[1] < width or (t.shape[1] > 1 and t.stride(1) != 1):
            raise ValueError(f"{name} must be {rows} rows of at least {width} bytes, row-major")
        if t.device != a.device:
            raise ValueError(f"{name} must be on a's device")
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.float16
    if out_dtype not in (torch.float16, torch.float32):
        raise TypeError("out_dtype must be torch.float16 or torch.float32")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    elif out.dtype != out_dtype or tuple(out.shape) != (M, N) or out.device != a.device:
        raise ValueError("out must be M×N on a's device with dtype out_dtype")
    if bias is not None and (bias.dtype != torch.float32 or bias.numel() != N or bias.dim() != 1
                             or bias.device != a.device or (N > 1 and bias.stride(0) != 1)):
        raise ValueError("bias must be a contiguous float32 CUDA tensor of N elements")
    if residual is not None:
        _check_operand(residual, "residual")
        if residual.dtype != torch.float16 or tuple(residual.shape) != (M, N) \
                or residual.device != a.device:
            raise ValueError("residual must be M×N float16 on a's device")
    epi = tg_epilogue_ex_t(TG_EPI_RELU if relu else TG_EPI_NONE,
                           TG_DTYPE_F32 if out_dtype == torch.float32 else TG_DTYPE_F16,
                           bias.data_ptr() if bias is not None else None,
                           residual.data_ptr() if residual is not None else None,
                           _ld(residual) if residual is not None else 0)
    ldb = lambda t: int(t.stride(0)) if t.shape[0] > 1 else (int(t.shape[1]) + 15) // 16 * 16  # noqa
    with torch.cuda.device(a.device):
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        st = tg_gemm_mxfp4(a.data_ptr(), bq.data_ptr(), bscale.data_ptr(), out.data_ptr(), M, N,
                           K, _ld(a), ldb(bq), ldb(bscale), _ld(out), epi, s.cuda_stream)
    if st != TG_OK:
        raise TgemmError(st, "tg_gemm_mxfp4")
    return out


def gemm_sp24(ac, e, b, relu: bool = False, out=None, stream=None, *, bias=None, residual=None,
              out_dtype=None):
    """C = out(act(A @ b + bias) + residual) with A 2:4 structured-sparse.

    ac: CUDA float16/bfloat16 tensor M × K/2 of kept values; e: CUDA int32 (or
    uint32 bits in int32) tensor M × K/32 of metadata words; b: K × N of ac's
    dtype.  Rows 16-byte aligned (row strides multiples of 8 elements, 4 words).
    bias, residual, out_dtype, out and stream as for ``gemm``.
    """
    import torch
    _check_operand(ac, "ac")
    _check_operand(b, "b")
    M, half = ac.shape
    K, N = b.shape
    if half * 2 != K or K % 32 != 0:
        raise ValueError("ac must be M × K/2 for b of K rows, K a multiple of 32")
    if ac.dtype != b.dtype:
        raise TypeError("ac and b must share a dtype")
    if not isinstance(e, torch.Tensor) or e.dtype != torch.int32 or e.dim() != 2 \
            or tuple(e.shape) != (M, K // 32) or (K > 32 and e.stride(1) != 1):
        raise ValueError("e must be an int32 tensor of M × K/32 metadata words")
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else ac.dtype
    if out_dtype not in (ac.dtype, torch.float32):
        raise TypeError(f"out_dtype must be {ac.dtype} or torch.float32")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=ac.device)
    in_code = TG_DTYPE_BF16 if ac.dtype == torch.bfloat16 else TG_DTYPE_F16
    epi = tg_epilogue_ex_t(TG_EPI_RELU if relu else TG_EPI_NONE,
                           TG_DTYPE_F32 if out_dtype == torch.float32 else in_code,
                           bias.data_ptr() if bias is not None else None,
                           residual.data_ptr() if residual is not None else None,
                           _ld(residual) if residual is not None else 0)
    lde = int(e.stride(0)) if M > 1 else max(4, (K // 32 + 3) // 4 * 4)
    with torch.cuda.device(ac.device):
        s = stream if stream is not None else torch.cuda.current_stream(ac.device)
        st = tg_gemm_sp24(in_code, ac.data_ptr(), e.data_ptr(), b.data_ptr(), out.data_ptr(), M,
                          N, K, _ld(ac), lde, _ld(b), _ld(out), epi, s.cuda_stream)
    if st != TG_OK:
        raise TgemmError(st, "tg_gemm_sp24")
    return out


def gemm_host(a, b, relu: bool = False, stream=None, device=None):
    """End-to-end C = epi(a @ b) from host (CPU) float16 tensors, through
    tg_gemm_f16_host: the library uploads a and B and downloads C block by
    block on its own copy streams, overlapped with the products.  Returns C
    in a pinned host tensor once it is complete.  Pinned a and b let the
    copies overlap; pageable ones work, without overlap.
    """
    import torch
    for t, name in ((a, "a"), (b, "b")):
        if t.device.type != "cpu" or t.dtype != torch.float16 or t.dim() != 2:
            raise ValueError(f"{name} must be a 2-D float16 CPU tensor")
        if t.stride(1) != 1:
            raise ValueError(f"{name} must have unit column stride")
    M, K = a.shape
    if b.shape[0] != K:
        raise ValueError(f"inner sizes differ: a is {tuple(a.shape)}, b is {tuple(b.shape)}")
    N = b.shape[1]
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    hc = torch.empty((M, N), dtype=torch.float16, pin_memory=True)
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        st = tg_gemm_f16_host(a.data_ptr(), b.data_ptr(), hc.data_ptr(), M, N, K,
                              max(a.stride(0), 1), max(b.stride(0), 1), max(N, 1),
                              TG_EPI_RELU if relu else TG_EPI_NONE, s.cuda_stream)
        if st != TG_OK:
            raise TgemmError(st, "tg_gemm_f16_host")
        st = tg_sync_status(s.cuda_stream)
        if st != TG_OK:
            raise TgemmError(st, "tg_sync_status")
    return hc


def sync_status(stream=None) -> None:
    """Wait for the stream and raise TgemmError if a kernel reported a timeout."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    st = tg_sync_status(s.cuda_stream)
    if st != TG_OK:
        raise TgemmError(st, "tg_sync_status")
