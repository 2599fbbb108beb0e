"""CPU oracle for C = epi(A·B) — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under test never imports,
links or calls it; the two share no code.

The arithmetic lives in ``tgemm_oracle.c`` (plain C, fp64 accumulation, one
round-to-nearest-even to fp16).  This module builds it with gcc on first use
and wraps it with ctypes.  See that file's header for the passages it follows
and the readings it takes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "tgemm_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_default = None


def compile_source(src: str, out: str) -> str:
    """gcc-compile one C file into a shared library (OpenMP when available)."""
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle next to its source. Returns the .so path."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(SOURCE)):
            return _LIB
        return compile_source(SOURCE, _LIB)


def _ptr(a, ct):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ct))


def _as_u16(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("expected float16 or uint16 bits")
    return np.ascontiguousarray(x)


class Oracle:
    """ctypes view of one build of ``tgemm_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.oracle_gemm_f16.argtypes = [u16p, u16p, u16p, f64p, i64, i64, i64, i64, i64, i64,
                                        ctypes.c_int]
        lib.oracle_gemm_f16.restype = ctypes.c_int
        lib.oracle_gemm_f16_at.argtypes = [u16p, u16p, i64, i64, i64, ctypes.c_int, i64p, i64p,
                                           i64, u16p, f64p]
        lib.oracle_gemm_f16_at.restype = ctypes.c_int
        lib.oracle_f16_from_f64_array.argtypes = [f64p, u16p, i64]
        lib.oracle_f64_from_f16_array.argtypes = [u16p, f64p, i64]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_gemm_bf16.argtypes = lib.oracle_gemm_f16.argtypes
        lib.oracle_gemm_bf16.restype = ctypes.c_int
        lib.oracle_gemm_bf16_at.argtypes = lib.oracle_gemm_f16_at.argtypes
        lib.oracle_gemm_bf16_at.restype = ctypes.c_int
        lib.oracle_bf16_from_f64_array.argtypes = [f64p, u16p, i64]
        lib.oracle_f64_from_bf16_array.argtypes = [u16p, f64p, i64]
        f32p = ctypes.POINTER(ctypes.c_float)
        vp = ctypes.c_void_p
        lib.oracle_gemm_ex.argtypes = [ctypes.c_int, ctypes.c_int, u16p, u16p, vp, f64p, i64, i64,
                                       i64, i64, i64, i64, ctypes.c_int, f32p, u16p, i64]
        lib.oracle_gemm_ex.restype = ctypes.c_int
        lib.oracle_gemm_ex_at.argtypes = [ctypes.c_int, ctypes.c_int, u16p, u16p, i64, i64, i64,
                                          ctypes.c_int, f32p, u16p, i64, i64p, i64p, i64, vp,
                                          f64p]
        lib.oracle_gemm_ex_at.restype = ctypes.c_int
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_f64_from_e2m1.argtypes = [ctypes.c_uint8]
        lib.oracle_f64_from_e2m1.restype = ctypes.c_double
        lib.oracle_f64_from_e8m0.argtypes = [ctypes.c_uint8]
        lib.oracle_f64_from_e8m0.restype = ctypes.c_double
        lib.oracle_mxfp4_dequant_f16.argtypes = [u8p, i64, u8p, i64, i64, i64, u16p, i64]
        lib.oracle_mxfp4_dequant_f16.restype = ctypes.c_int
        u32p = ctypes.POINTER(ctypes.c_uint32)
        lib.oracle_sp24_decompress.argtypes = [u16p, i64, u32p, i64, i64, i64, u16p, i64]
        lib.oracle_sp24_decompress.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def f16_from_f64(self, x) -> np.ndarray:
        """Round float64 values to binary16 bits (RNE), element-wise."""
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f16_from_f64_array(_ptr(x, ctypes.c_double),
                                           _ptr(out, ctypes.c_uint16), x.size)
        return out

    def f64_from_f16(self, h) -> np.ndarray:
        """Decode binary16 bits to float64, element-wise."""
        h = _as_u16(np.asarray(h))
        out = np.empty(h.shape, dtype=np.float64)
        self.lib.oracle_f64_from_f16_array(_ptr(h, ctypes.c_uint16),
                                           _ptr(out, ctypes.c_double), h.size)
        return out

    def bf16_from_f64(self, x) -> np.ndarray:
        """Round float64 values to bfloat16 bits (RNE), element-wise."""
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_bf16_from_f64_array(_ptr(x, ctypes.c_double),
                                            _ptr(out, ctypes.c_uint16), x.size)
        return out

    def f64_from_bf16(self, h) -> np.ndarray:
        """Decode bfloat16 bits (uint16) to float64, element-wise."""
        h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16))
        out = np.empty(h.shape, dtype=np.float64)
        self.lib.oracle_f64_from_bf16_array(_ptr(h, ctypes.c_uint16),
                                            _ptr(out, ctypes.c_double), h.size)
        return out

    def gemm(self, A: np.ndarray, B: np.ndarray, M: int, N: int, K: int,
             relu: bool = False, want_ref: bool = False, dtype: str = "f16"):
        """Full product of A (M×lda, lda ≥ K) and B (K×ldb, ldb ≥ N).

        dtype "f16": A and B are float16 (or their bits); returns C as float16.
        dtype "bf16": A and B are bfloat16 bit patterns (uint16); returns C as
        bfloat16 bits (uint16).  With ``want_ref`` also returns the fp64 values
        epi(sum) before rounding (M×N).
        """
        A = _as_u16(A)
        B = _as_u16(B)
        lda = A.shape[1] if A.ndim == 2 else K
        ldb = B.shape[1] if B.ndim == 2 else N
        C = np.empty((M, N), dtype=np.uint16)
        ref = np.empty((M, N), dtype=np.float64) if want_ref else None
        fn = self.lib.oracle_gemm_bf16 if dtype == "bf16" else self.lib.oracle_gemm_f16
        rc = fn(_ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16), _ptr(C, ctypes.c_uint16),
                _ptr(ref, ctypes.c_double), M, N, K, lda, ldb, N, int(bool(relu)))
        if rc != 0:
            raise ValueError("oracle gemm rejected its arguments")
        if dtype != "bf16":
            C = C.view(np.float16)
        return (C, ref) if want_ref else C

    def gemm_at(self, A: np.ndarray, B: np.ndarray, K: int, rows, cols, relu: bool = False,
                dtype: str = "f16"):
        """Selected elements (rows[t], cols[t]) of the same product.

        Returns (rounded values: float16, or bfloat16 bits for dtype "bf16";
        float64 values before rounding).
        """
        A = _as_u16(A)
        B = _as_u16(B)
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        n = rows.size
        out16 = np.empty(n, dtype=np.uint16)
        out64 = np.empty(n, dtype=np.float64)
        fn = self.lib.oracle_gemm_bf16_at if dtype == "bf16" else self.lib.oracle_gemm_f16_at
        rc = fn(_ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16), K, A.shape[1], B.shape[1],
                int(bool(relu)), _ptr(rows, ctypes.c_int64), _ptr(cols, ctypes.c_int64), n,
                _ptr(out16, ctypes.c_uint16), _ptr(out64, ctypes.c_double))
        if rc != 0:
            raise ValueError("oracle gemm_at rejected its arguments")
        return (out16 if dtype == "bf16" else out16.view(np.float16)), out64


_FMT = {"f16": 0, "bf16": 1, "f32": 2}


def _ex_outputs(out_dtype: str, shape):
    if out_dtype == "f32":
        return np.empty(shape, dtype=np.float32)
    return np.empty(shape, dtype=np.uint16)


def _ex_view(C, out_dtype: str):
    return C.view(np.float16) if out_dtype == "f16" else C


def _gemm_ex(self, A, B, M, N, K, relu=False, bias=None, R=None, in_dtype="f16",
             out_dtype="f16", want_ref=False):
    """C = out_round(act(A·B + bias[j]) + R[i][j]) (see tgemm_oracle.c).

    A, B, R: float16 arrays or 16-bit patterns of ``in_dtype`` ("f16"/"bf16");
    bias: float32 vector of N or None; R: M×ldr or None.  Returns C as
    float16 (out "f16"), bfloat16 bits (out "bf16") or float32 (out "f32").
    """
    A = _as_u16(A)
    B = _as_u16(B)
    lda = A.shape[1] if A.ndim == 2 else K
    ldb = B.shape[1] if B.ndim == 2 else N
    bias_a = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float32))
    R_a = None if R is None else _as_u16(np.asarray(R))
    ldr = 0 if R_a is None else R_a.shape[1]
    C = _ex_outputs(out_dtype, (M, N))
    ref = np.empty((M, N), dtype=np.float64) if want_ref else None
    rc = self.lib.oracle_gemm_ex(_FMT[in_dtype], _FMT[out_dtype], _ptr(A, ctypes.c_uint16),
                                 _ptr(B, ctypes.c_uint16), C.ctypes.data_as(ctypes.c_void_p),
                                 _ptr(ref, ctypes.c_double), M, N, K, lda, ldb, N,
                                 int(bool(relu)), _ptr(bias_a, ctypes.c_float),
                                 _ptr(R_a, ctypes.c_uint16), ldr)
    if rc != 0:
        raise ValueError("oracle_gemm_ex rejected its arguments")
    C = _ex_view(C, out_dtype)
    return (C, ref) if want_ref else C


def _gemm_ex_at(self, A, B, K, rows, cols, relu=False, bias=None, R=None, in_dtype="f16",
                out_dtype="f16"):
    """Selected elements of gemm_ex; returns (rounded values, fp64 values)."""
    A = _as_u16(A)
    B = _as_u16(B)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    bias_a = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float32))
    R_a = None if R is None else _as_u16(np.asarray(R))
    ldr = 0 if R_a is None else R_a.shape[1]
    out = _ex_outputs(out_dtype, rows.size)
    out64 = np.empty(rows.size, dtype=np.float64)
    rc = self.lib.oracle_gemm_ex_at(_FMT[in_dtype], _FMT[out_dtype], _ptr(A, ctypes.c_uint16),
                                    _ptr(B, ctypes.c_uint16), K, A.shape[1], B.shape[1],
                                    int(bool(relu)), _ptr(bias_a, ctypes.c_float),
                                    _ptr(R_a, ctypes.c_uint16), ldr, _ptr(rows, ctypes.c_int64),
                                    _ptr(cols, ctypes.c_int64), rows.size,
                                    out.ctypes.data_as(ctypes.c_void_p),
                                    _ptr(out64, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_gemm_ex_at rejected its arguments")
    return _ex_view(out, out_dtype), out64


Oracle.gemm_ex = _gemm_ex
Oracle.gemm_ex_at = _gemm_ex_at


def gemm_ex(*args, **kw):
    return default().gemm_ex(*args, **kw)


def gemm_ex_at(*args, **kw):
    return default().gemm_ex_at(*args, **kw)


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def num_threads() -> int:
    return default().num_threads()


def f16_from_f64(x) -> np.ndarray:
    return default().f16_from_f64(x)


def f64_from_f16(h) -> np.ndarray:
    return default().f64_from_f16(h)


def bf16_from_f64(x) -> np.ndarray:
    return default().bf16_from_f64(x)


def f64_from_bf16(h) -> np.ndarray:
    return default().f64_from_bf16(h)


def gemm(A, B, M, N, K, relu=False, want_ref=False, dtype="f16"):
    return default().gemm(A, B, M, N, K, relu, want_ref, dtype)


def gemm_at(A, B, K, rows, cols, relu=False, dtype="f16"):
    return default().gemm_at(A, B, K, rows, cols, relu, dtype)


def ulp_bf16(x) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x|: 2^(floor(log2|x|) - 7) for normal
    magnitudes, 2^-133 below the smallest normal (and at zero)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    out = np.full(a.shape, 2.0 ** -133)
    nz = a >= 2.0 ** -126
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    out[nz] = np.exp2(e[nz] - 7.0)
    return out


def ulp16(x) -> np.ndarray:
    """Spacing of binary16 numbers at |x|: 2^(floor(log2|x|) - 10) for normal
    magnitudes, 2^-24 below the smallest normal (and at zero)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    out = np.full(a.shape, 2.0 ** -24)
    nz = a >= 2.0 ** -14
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    out[nz] = np.exp2(e[nz] - 10.0)
    return out


# ------------------------------------------------------------------ MXFP4 weights

def _mx_e2m1(self, code: int) -> float:
    """Value of one 4-bit FP4 E2M1 code."""
    return float(self.lib.oracle_f64_from_e2m1(int(code) & 15))


def _mx_e8m0(self, x: int) -> float:
    """Value of one E8M0 scale byte: 2^(x - 127), NaN for 255."""
    return float(self.lib.oracle_f64_from_e8m0(int(x) & 255))


def _mxfp4_dequant(self, Bq, S, K, N):
    """Bdeq = fp16_rne(e2m1(code) * 2^(X - 127)) as a K×N float16 array.

    Bq: uint8, N rows of packed codes along k (row stride Bq.shape[1] >=
    ceil(K/2)); S: uint8 E8M0 scales, ceil(K/32) rows (row stride S.shape[1]
    >= N)."""
    Bq = np.ascontiguousarray(np.asarray(Bq, dtype=np.uint8))
    S = np.ascontiguousarray(np.asarray(S, dtype=np.uint8))
    out = np.empty((K, N), dtype=np.uint16)
    ldbq = Bq.shape[1] if Bq.ndim == 2 else (K + 1) // 2
    lds = S.shape[1] if S.ndim == 2 else N
    rc = self.lib.oracle_mxfp4_dequant_f16(_ptr(Bq, ctypes.c_uint8), ldbq,
                                          _ptr(S, ctypes.c_uint8), lds, K, N,
                                          _ptr(out, ctypes.c_uint16), N)
    if rc != 0:
        raise ValueError("oracle_mxfp4_dequant_f16 rejected its arguments")
    return out.view(np.float16)


def _gemm_mxfp4(self, A, Bq, S, M, N, K, relu=False, bias=None, R=None, out_dtype="f16"):
    """C = out(act(A·Bdeq + bias) + R) with Bdeq the dequantised MXFP4 weights
    (see tgemm_oracle.c); A and R fp16."""
    Bd = self.mxfp4_dequant(Bq, S, K, N)
    return self.gemm_ex(A, Bd, M, N, K, relu=relu, bias=bias, R=R, in_dtype="f16",
                        out_dtype=out_dtype)


def _gemm_mxfp4_at(self, A, Bq, S, K, N, rows, cols, relu=False, bias=None, R=None,
                   out_dtype="f16"):
    """Selected outputs of gemm_mxfp4; returns (rounded values, fp64 values)."""
    Bd = self.mxfp4_dequant(Bq, S, K, N)
    return self.gemm_ex_at(A, Bd, K, rows, cols, relu=relu, bias=bias, R=R, in_dtype="f16",
                           out_dtype=out_dtype)


Oracle.e2m1 = _mx_e2m1
Oracle.e8m0 = _mx_e8m0
Oracle.mxfp4_dequant = _mxfp4_dequant
Oracle.gemm_mxfp4 = _gemm_mxfp4
Oracle.gemm_mxfp4_at = _gemm_mxfp4_at


def mxfp4_dequant(*args, **kw):
    return default().mxfp4_dequant(*args, **kw)


def gemm_mxfp4(*args, **kw):
    return default().gemm_mxfp4(*args, **kw)


def gemm_mxfp4_at(*args, **kw):
    return default().gemm_mxfp4_at(*args, **kw)


# ------------------------------------------------------------------ 2:4 sparse A

def _sp24_decompress(self, Ac, E, M, K):
    """Dense A (M×K 16-bit patterns) from compressed values Ac (M rows of >= K/2
    16-bit patterns) and metadata E (M rows of >= K/32 uint32 words); see
    tgemm_oracle.c for the format.  Raises ValueError on invalid metadata."""
    Ac = _as_u16(np.asarray(Ac)) if np.asarray(Ac).dtype != np.uint16 else np.ascontiguousarray(Ac)
    E = np.ascontiguousarray(np.asarray(E, dtype=np.uint32))
    A = np.full((M, K), 0x7E00, dtype=np.uint16)  # NaN pattern: every element must be written
    rc = self.lib.oracle_sp24_decompress(_ptr(Ac, ctypes.c_uint16), Ac.shape[1],
                                        _ptr(E, ctypes.c_uint32), E.shape[1], M, K,
                                        _ptr(A, ctypes.c_uint16), K)
    if rc == -2:
        raise ValueError("sp24 metadata: a group's positions are not first < second")
    if rc != 0:
        raise ValueError("oracle_sp24_decompress rejected its arguments")
    return A


def _gemm_sp24(self, Ac, E, B, M, N, K, relu=False, bias=None, R=None, in_dtype="f16",
               out_dtype=None):
    """C = out(act(A·B + bias) + R) with A the 2:4 sparse matrix (Ac, E)."""
    A = self.sp24_decompress(Ac, E, M, K)
    return self.gemm_ex(A, B, M, N, K, relu=relu, bias=bias, R=R, in_dtype=in_dtype,
                        out_dtype=out_dtype or in_dtype)


def _gemm_sp24_at(self, Ac, E, B, K, rows, cols, relu=False, bias=None, R=None,
                  in_dtype="f16", out_dtype=None):
    """Selected outputs of gemm_sp24 (decompresses only the rows needed)."""
    rows = np.asarray(rows, dtype=np.int64)
    uniq, inv = np.unique(rows, return_inverse=True)
    Ac = np.asarray(Ac)
    A = self.sp24_decompress(Ac[uniq], np.asarray(E)[uniq], uniq.size, K)
    Rsub = None if R is None else np.asarray(R)[uniq]
    return self.gemm_ex_at(A, B, K, inv, cols, relu=relu, bias=bias, R=Rsub,
                           in_dtype=in_dtype, out_dtype=out_dtype or in_dtype)


Oracle.sp24_decompress = _sp24_decompress
Oracle.gemm_sp24 = _gemm_sp24
Oracle.gemm_sp24_at = _gemm_sp24_at


def sp24_decompress(*args, **kw):
    return default().sp24_decompress(*args, **kw)


def gemm_sp24(*args, **kw):
    return default().gemm_sp24(*args, **kw)


def gemm_sp24_at(*args, **kw):
    return default().gemm_sp24_at(*args, **kw)
