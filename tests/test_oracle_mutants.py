"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (no GPU).

Each C mutant is a textual edit of ``oracle/tgemm_oracle.c`` compiled into a
temporary library.  Each Python mutant is a textual edit of one function of
``oracle/__init__.py``, compiled in that module's namespace and installed on a
fresh ``Oracle`` (methods) or patched over the module attribute for the one
test (the tolerance spacings).  The committed oracle is never modified.
"""

import inspect
import os
import types

import pytest

import oracle
import oracle_pins

# (name, original text, replacement) — each edit must apply at least once.
# (A ReLU that lets -0 through is not listed: the fp64 sum starts at +0 and
# IEEE addition never turns it into -0, so that mutant is equivalent.)
MUTANTS = [
    ("drop_last_term", "k < K; ++k)", "k < K - 1; ++k)"),
    ("drop_first_term", "for (int64_t k = 0; k < K;", "for (int64_t k = 1; k < K;"),
    ("wrong_sign_first_product", "acc[j] += a * g_lut[brow[j]];",
     "acc[j] += (k == 0 ? -a : a) * g_lut[brow[j]];"),
    ("wrong_b_row", "const uint16_t* brow = B + k * ldb;",
     "const uint16_t* brow = B + ((k + 1) % K) * ldb;"),
    ("transposed_a", "double a = g_lut[A[i * lda + k]];",
     "double a = g_lut[A[(k % M) * lda + (i % K)]];"),
    ("truncating_round", "double frac = n - fl; /* exact */", "double frac = 0.0;"),
    ("ties_away", "return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    ("fp32_accumulator", "double* acc = (double*)malloc(sizeof(double)",
     "float* acc = (float*)malloc(sizeof(float)"),
    ("relu_as_abs", "if (relu) return v > 0.0 ? v : 0.0;", "if (relu) return fabs(v);"),
    ("relu_ignored", "if (relu) return v > 0.0 ? v : 0.0;", "if (relu) return v;"),
    ("flush_subnormals", "double n = round_half_even(ldexp(a, 24));", "double n = 0.0;"),
    ("late_overflow", "if (e > 15) return", "if (e > 16) return"),
    ("decode_bias", "e - 25);", "e - 24);"),
    ("decode_subnormal", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    ("ldb_ignored", "g_lut[bcol[k * ldb]]", "g_lut[bcol[k * (ldb - (ldb > 1))]]"),
    # bfloat16 variant
    ("bf16_decode_bias", "e - 134);", "e - 133);"),
    ("bf16_decode_subnormal", "v = ldexp((double)m, -133);", "v = ldexp((double)m, -134);"),
    ("bf16_flush_subnormals", "double n = round_half_even(ldexp(a, 133));", "double n = 0.0;"),
    ("bf16_late_overflow", "if (e > 127) return", "if (e > 128) return"),
    ("bf16_fp16_lut", "acc[j] += a * g_lut_bf16[brow[j]];", "acc[j] += a * g_lut[brow[j]];"),
    ("bf16_rounds_as_fp16", "C[i * ldc + j] = oracle_bf16_from_f64(v);",
     "C[i * ldc + j] = oracle_f16_from_f64(v);"),
    ("bf16_truncating_round", "double n = round_half_even(ldexp(a, 7 - e));",
     "double n = floor(ldexp(a, 7 - e));"),
    # extended epilogue
    ("ex_bias_after_relu", "    if (bias) v += (double)bias[j];\n    v = epi_apply(v, relu);",
     "    v = epi_apply(v, relu);\n    if (bias) v += (double)bias[j];"),
    ("ex_residual_before_relu",
     "    v = epi_apply(v, relu);\n    if (R) v += decode16(R[i * ldr + j], in_fmt);",
     "    if (R) v += decode16(R[i * ldr + j], in_fmt);\n    v = epi_apply(v, relu);"),
    ("ex_bias_by_row", "if (bias) v += (double)bias[j];", "if (bias) v += (double)bias[i];"),
    ("ex_residual_ignored", "if (R) v += decode16(R[i * ldr + j], in_fmt);", "(void)R;"),
    ("ex_residual_row_ignored", "decode16(R[i * ldr + j], in_fmt)",
     "decode16(R[(i % 1) * ldr + j], in_fmt)"),
    ("ex_f32_through_f16", "if (out_fmt == 2) ((float*)C)[idx] = (float)v;",
     "if (out_fmt == 2) ((float*)C)[idx] = (float)oracle_f64_from_f16(oracle_f16_from_f64(v));"),
    # MXFP4 weights
    ("mx_nibbles_swapped", "(k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15)",
     "(k & 1) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4)"),
    ("mx_scale_block_16", "S[(k / 32) * lds + n]", "S[(k / 16) * lds + n]"),
    ("mx_scale_by_row", "S[(k / 32) * lds + n]", "S[(n / 32) * lds + k % lds]"),
    ("mx_e2m1_bias_2", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)"),
    ("mx_e2m1_no_subnormal", "(e == 0) ? ldexp((double)m, -1)", "(e == 0) ? ldexp(1.0 + 0.5 * m, -1)"),
    ("mx_e2m1_sign_ignored", "return s ? -mag : mag;", "return mag;"),
    ("mx_e8m0_bias_128", "return ldexp(1.0, (int)x - 127);", "return ldexp(1.0, (int)x - 128);"),
    ("mx_e8m0_nan_ignored", "if (x == 255) return NAN;", "if (x == 256) return NAN;"),
    ("mx_deq_no_rounding", "Bdeq[k * ldb + n] = oracle_f16_from_f64(v);",
     "Bdeq[k * ldb + n] = oracle_f16_from_f64(v) & 0xFFFE;"),
    # 2:4 sparse A
    ("sp24_position_fields_swapped", "uint32_t p0 = nib & 3u, p1 = (nib >> 2) & 3u;",
     "uint32_t p1 = nib & 3u, p0 = (nib >> 2) & 3u;"),
    ("sp24_group_order_reversed", "(word >> (4 * (G % 8))) & 15u", "(word >> (4 * (7 - G % 8))) & 15u"),
    ("sp24_values_swapped", "A[i * lda + 4 * G + p0] = Ac[i * ldac + 2 * G];",
     "A[i * lda + 4 * G + p0] = Ac[i * ldac + 2 * G + 1];"),
    ("sp24_word_per_16k", "E[i * lde + G / 8]", "E[i * lde + G / 16]"),
    ("sp24_no_zero_fill", "for (int64_t k = 0; k < K; ++k) A[i * lda + k] = 0;", "(void)0;"),
    ("sp24_order_unchecked", "if (p0 >= p1) return -2;", "(void)0;"),
]


def _pin_catches(o):
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failures.append(pin.__name__)
        except (ValueError, FloatingPointError, OverflowError):
            failures.append(pin.__name__ + "(raised)")
    return failures


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = os.path.join(str(tmp_path), f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, os.path.join(str(tmp_path), f"lib{name}.so"))
    caught = _pin_catches(oracle.Oracle(lib))
    assert caught, f"mutant {name} passed every pin"


# Python-level parts of the oracle: (name, function, original text, replacement).
# The spacing functions set the parity tolerance; the *_at functions produce
# the expected values of the large sampled GPU tests.
PY_MUTANTS = [
    ("ulp_bf16_mantissa_8", "ulp_bf16", "e[nz] - 7.0", "e[nz] - 8.0"),
    ("ulp_bf16_normal_from_2^-127", "ulp_bf16", "a >= 2.0 ** -126", "a >= 2.0 ** -127"),
    ("ulp_bf16_subnormal_2^-134", "ulp_bf16", "np.full(a.shape, 2.0 ** -133)",
     "np.full(a.shape, 2.0 ** -134)"),
    ("ulp16_mantissa_11", "ulp16", "e[nz] - 10.0", "e[nz] - 11.0"),
    ("ulp16_normal_from_2^-15", "ulp16", "a >= 2.0 ** -14", "a >= 2.0 ** -15"),
    ("sp24_at_inverse_sorted", "_gemm_sp24_at", "gemm_ex_at(A, B, K, inv,",
     "gemm_ex_at(A, B, K, np.sort(inv),"),
    ("sp24_at_residual_not_subset", "_gemm_sp24_at", "np.asarray(R)[uniq]", "np.asarray(R)"),
    ("sp24_at_metadata_not_subset", "_gemm_sp24_at", "np.asarray(E)[uniq]",
     "np.asarray(E)[:uniq.size]"),
    ("sp24_at_out_type_ignored", "_gemm_sp24_at", "out_dtype=out_dtype or in_dtype",
     "out_dtype=in_dtype"),
    ("mx_at_relu_dropped", "_gemm_mxfp4_at", "rows, cols, relu=relu,", "rows, cols, relu=False,"),
    ("mx_at_bias_dropped", "_gemm_mxfp4_at", "bias=bias, R=R, in_dtype", "bias=None, R=R, in_dtype"),
    ("mx_at_residual_dropped", "_gemm_mxfp4_at", "R=R, in_dtype", "R=None, in_dtype"),
]

_METHODS = {"_gemm_sp24_at": "gemm_sp24_at", "_gemm_mxfp4_at": "gemm_mxfp4_at"}


def _mutated(fname, old, new):
    src = inspect.getsource(getattr(oracle, fname))
    assert src.count(old) >= 1, f"mutation site {old!r} not found in {fname}"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant of {fname}>", "exec"), ns)
    return ns[fname]


@pytest.mark.parametrize("name,fname,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_python_mutant_is_caught(monkeypatch, name, fname, old, new):
    fn = _mutated(fname, old, new)
    o = oracle.Oracle(oracle.build())
    if fname in _METHODS:
        setattr(o, _METHODS[fname], types.MethodType(fn, o))
    else:
        monkeypatch.setattr(oracle, fname, fn)
    caught = _pin_catches(o)
    assert caught, f"mutant {name} passed every pin"
