/*
 * CPU oracle for the tiled FP16 GEMM — TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline may load this file's library.  The product path (libtgemm) never
 * links, loads or calls it, and the two share no code.
 *
 * What it computes (the plain definition of the operation):
 *
 *   C[i][j] = fp16_rne( epi( sum_{k<K} (double)A[i][k] * (double)B[k][j] ) )
 *
 *   - "5分钟上手TileLang" (0539edu.com), section "安装与第一个内核": the
 *     quickstart kernel computes C (M×N, fp16) from A (M×K, fp16) and
 *     B (K×N, fp16), both row-major, with a float32 fragment accumulator.
 *   - same page, section "避坑与调参": the accumulator stays in float32 and
 *     the cast to fp16 happens once, at the final copy.
 *   - "TileLang：比 Triton 低一层的 tile 语言" (anrans.github.io), section
 *     "第一个 kernel：GEMM": the same kernel with block_K = 64.
 *   - "TileLang：让GPU编程像Python一样简单的高性能计算新范式" (coreui.cn),
 *     the ReLU epilogue: max(C_local, 0) is applied to the float32
 *     accumulator before the copy to the fp16 output.
 *
 * Readings taken where the pages are silent:
 *   - the reference sum is carried in fp64 (each fp16×fp16 product is exact
 *     in fp64; the fp64 sum over K ≤ 8192 is far below one fp16 ulp off the
 *     exact value), in k-ascending order;
 *   - the rounding to fp16 is round-to-nearest, ties-to-even, done once from
 *     fp64; overflow goes to ±inf; subnormals are kept;
 *   - epi(x) = x > 0 ? x : +0 for ReLU (so -0 and NaN map to +0), epi(x) = x
 *     otherwise.
 *
 * Loop order i-k-j with an fp64 row accumulator, OpenMP over rows (when the
 * compiler offers it).  No blocking, no reordering of the k sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- binary16 <-> binary64 (IEEE 754-2008 binary16 layout: 1|5|10, bias 15) */

double oracle_f64_from_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24); /* subnormal: m · 2^-24 */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1.m) · 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a non-negative double that is an exact multiple of 2^-k to the
 * nearest integer, ties to even.  n is representable (|n| < 2^53). */
static double round_half_even(double n)
{
    double fl = floor(n);
    double frac = n - fl; /* exact */
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    /* tie */
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint16_t oracle_f16_from_f64(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24; n in [0, 1024] (1024 = min normal) */
        double n = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)n);
    }
    int E;
    frexp(a, &E);          /* a = f · 2^E, f in [0.5, 1) */
    int e = E - 1;         /* a in [2^e, 2^(e+1)) */
    double n = round_half_even(ldexp(a, 10 - e)); /* in [1024, 2048] */
    if (n == 2048.0) {
        n = 1024.0;
        e += 1;
    }
    if (e > 15) return (uint16_t)(sign | 0x7c00); /* overflow -> inf */
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(n - 1024.0));
}

void oracle_f16_from_f64_array(const double* x, uint16_t* h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = oracle_f16_from_f64(x[i]);
}

void oracle_f64_from_f16_array(const uint16_t* h, double* x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) x[i] = oracle_f64_from_f16(h[i]);
}

static double g_lut[65536];
static int g_lut_ready = 0;

static void lut_init(void)
{
    if (g_lut_ready) return;
    for (int i = 0; i < 65536; ++i) g_lut[i] = oracle_f64_from_f16((uint16_t)i);
    g_lut_ready = 1;
}

static double epi_apply(double v, int relu)
{
    if (relu) return v > 0.0 ? v : 0.0;
    return v;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full product.  A: M×K with row stride lda, B: K×N with row stride ldb,
 * C: M×N with row stride ldc (fp16 bits).  If Cref is not NULL it receives the
 * fp64 value epi(sum) before rounding, densely as M×N.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_gemm_f16(const uint16_t* A, const uint16_t* B, uint16_t* C, double* Cref,
                    int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                    int relu)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N) return -1;
    lut_init();
    int err = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!acc) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < M; ++i) {
            if (!acc) continue;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = g_lut[A[i * lda + k]];
                const uint16_t* brow = B + k * ldb;
                for (int64_t j = 0; j < N; ++j) acc[j] += a * g_lut[brow[j]];
            }
            for (int64_t j = 0; j < N; ++j) {
                double v = epi_apply(acc[j], relu);
                C[i * ldc + j] = oracle_f16_from_f64(v);
                if (Cref) Cref[i * N + j] = v;
            }
        }
        free(acc);
    }
    return err ? -1 : 0;
}

/*
 * Selected outputs only: for each t < n, the element (rows[t], cols[t]) of the
 * same product, computed as one k-ascending fp64 dot product (the same order
 * as the full routine, so the two agree bit for bit).
 */
int oracle_gemm_f16_at(const uint16_t* A, const uint16_t* B, int64_t K, int64_t lda,
                       int64_t ldb, int relu, const int64_t* rows, const int64_t* cols,
                       int64_t n, uint16_t* out16, double* out64)
{
    if (K < 0 || lda < K) return -1;
    lut_init();
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t* arow = A + rows[t] * lda;
        const uint16_t* bcol = B + cols[t];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += g_lut[arow[k]] * g_lut[bcol[k * ldb]];
        double v = epi_apply(s, relu);
        if (out16) out16[t] = oracle_f16_from_f64(v);
        if (out64) out64[t] = v;
    }
    return 0;
}

/* ========================================================================
 * bfloat16 variant.  The pages define the GEMM for fp16 storage only; the
 * bf16 variant applies the same definition with bfloat16 storage of A, B and
 * C:  C[i][j] = bf16_rne( epi( sum_k (double)A[i][k] * (double)B[k][j] ) ).
 * bfloat16 is the upper half of an IEEE binary32: 1 sign bit, 8 exponent
 * bits (bias 127), 7 fraction bits; subnormal spacing 2^-133; largest finite
 * value (2 - 2^-7) * 2^127.  Rounding is once, from fp64, ties to even.
 * ======================================================================== */

double oracle_f64_from_bf16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int m = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -133); /* subnormal: m · 2^-133 */
    } else if (e == 255) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + m), e - 134); /* (1.m) · 2^(e-127) */
    }
    return sign ? -v : v;
}

uint16_t oracle_bf16_from_f64(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7fc0);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7f80);
    if (a < ldexp(1.0, -126)) {
        /* subnormal range: quantum 2^-133; n in [0, 128] (128 = min normal) */
        double n = round_half_even(ldexp(a, 133));
        return (uint16_t)(sign | (uint16_t)n);
    }
    int E;
    frexp(a, &E);
    int e = E - 1; /* a in [2^e, 2^(e+1)) */
    double n = round_half_even(ldexp(a, 7 - e)); /* in [128, 256] */
    if (n == 256.0) {
        n = 128.0;
        e += 1;
    }
    if (e > 127) return (uint16_t)(sign | 0x7f80); /* overflow -> inf */
    return (uint16_t)(sign | (uint16_t)((e + 127) << 7) | (uint16_t)(n - 128.0));
}

void oracle_bf16_from_f64_array(const double* x, uint16_t* h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = oracle_bf16_from_f64(x[i]);
}

void oracle_f64_from_bf16_array(const uint16_t* h, double* x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) x[i] = oracle_f64_from_bf16(h[i]);
}

static double g_lut_bf16[65536];
static int g_lut_bf16_ready = 0;

static void lut_bf16_init(void)
{
    if (g_lut_bf16_ready) return;
    for (int i = 0; i < 65536; ++i) g_lut_bf16[i] = oracle_f64_from_bf16((uint16_t)i);
    g_lut_bf16_ready = 1;
}

/* Full product, bf16 storage; arguments as oracle_gemm_f16. */
int oracle_gemm_bf16(const uint16_t* A, const uint16_t* B, uint16_t* C, double* Cref,
                     int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                     int relu)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N) return -1;
    lut_bf16_init();
    int err = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!acc) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < M; ++i) {
            if (!acc) continue;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = g_lut_bf16[A[i * lda + k]];
                const uint16_t* brow = B + k * ldb;
                for (int64_t j = 0; j < N; ++j) acc[j] += a * g_lut_bf16[brow[j]];
            }
            for (int64_t j = 0; j < N; ++j) {
                double v = epi_apply(acc[j], relu);
                C[i * ldc + j] = oracle_bf16_from_f64(v);
                if (Cref) Cref[i * N + j] = v;
            }
        }
        free(acc);
    }
    return err ? -1 : 0;
}

/* Selected outputs, bf16 storage; arguments as oracle_gemm_f16_at. */
int oracle_gemm_bf16_at(const uint16_t* A, const uint16_t* B, int64_t K, int64_t lda,
                        int64_t ldb, int relu, const int64_t* rows, const int64_t* cols,
                        int64_t n, uint16_t* out16, double* out64)
{
    if (K < 0 || lda < K) return -1;
    lut_bf16_init();
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t* arow = A + rows[t] * lda;
        const uint16_t* bcol = B + cols[t];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += g_lut_bf16[arow[k]] * g_lut_bf16[bcol[k * ldb]];
        double v = epi_apply(s, relu);
        if (out16) out16[t] = oracle_bf16_from_f64(v);
        if (out64) out64[t] = v;
    }
    return 0;
}

/* ========================================================================
 * Extended epilogue.  The pages show the ReLU epilogue as an element-wise
 * step on the fp32 accumulator before the final copy ("TileLang：让GPU编程像
 * Python一样简单的高性能计算新范式", T.Parallel over C_local); the same step
 * here also adds a per-column bias and a residual matrix and may keep the
 * result in fp32.  Reading taken (stated in the design notes):
 *
 *   C[i][j] = out_round( act( sum_k A[i][k]·B[k][j] + bias[j] ) + R[i][j] )
 *
 * with the sum in fp64 (k ascending), bias an fp32 vector over columns (or
 * absent), R a matrix in the input storage type with row stride ldr (or
 * absent), act = ReLU or identity, and out_round one rounding to fp16, bf16
 * or binary32.
 *   in_fmt:  0 = fp16 inputs (A, B, R), 1 = bf16
 *   out_fmt: 0 = fp16, 1 = bf16, 2 = fp32 (C is float*)
 * ======================================================================== */

static double decode16(uint16_t h, int fmt) { return fmt ? g_lut_bf16[h] : g_lut[h]; }

static double ex_value(double s, int64_t i, int64_t j, int relu, const float* bias,
                       const uint16_t* R, int64_t ldr, int in_fmt)
{
    double v = s;
    if (bias) v += (double)bias[j];
    v = epi_apply(v, relu);
    if (R) v += decode16(R[i * ldr + j], in_fmt);
    return v;
}

static void ex_store(void* C, int64_t idx, double v, int out_fmt)
{
    if (out_fmt == 2) ((float*)C)[idx] = (float)v; /* IEEE binary32, round to nearest even */
    else if (out_fmt == 1) ((uint16_t*)C)[idx] = oracle_bf16_from_f64(v);
    else ((uint16_t*)C)[idx] = oracle_f16_from_f64(v);
}

int oracle_gemm_ex(int in_fmt, int out_fmt, const uint16_t* A, const uint16_t* B, void* C,
                   double* Cref, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                   int64_t ldc, int relu, const float* bias, const uint16_t* R, int64_t ldr)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N) return -1;
    if (R && ldr < N) return -1;
    if (in_fmt < 0 || in_fmt > 1 || out_fmt < 0 || out_fmt > 2) return -1;
    lut_init();
    lut_bf16_init();
    int err = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!acc) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < M; ++i) {
            if (!acc) continue;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = decode16(A[i * lda + k], in_fmt);
                const uint16_t* brow = B + k * ldb;
                for (int64_t j = 0; j < N; ++j) acc[j] += a * decode16(brow[j], in_fmt);
            }
            for (int64_t j = 0; j < N; ++j) {
                double v = ex_value(acc[j], i, j, relu, bias, R, ldr, in_fmt);
                ex_store(C, i * ldc + j, v, out_fmt);
                if (Cref) Cref[i * N + j] = v;
            }
        }
        free(acc);
    }
    return err ? -1 : 0;
}

int oracle_gemm_ex_at(int in_fmt, int out_fmt, const uint16_t* A, const uint16_t* B, int64_t K,
                      int64_t lda, int64_t ldb, int relu, const float* bias, const uint16_t* R,
                      int64_t ldr, const int64_t* rows, const int64_t* cols, int64_t n,
                      void* out, double* out64)
{
    if (K < 0 || lda < K || in_fmt < 0 || in_fmt > 1 || out_fmt < 0 || out_fmt > 2) return -1;
    lut_init();
    lut_bf16_init();
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t* arow = A + rows[t] * lda;
        const uint16_t* bcol = B + cols[t];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += decode16(arow[k], in_fmt) * decode16(bcol[k * ldb], in_fmt);
        double v = ex_value(s, rows[t], cols[t], relu, bias, R, ldr, in_fmt);
        if (out) ex_store(out, t, v, out_fmt);
        if (out64) out64[t] = v;
    }
    return 0;
}

/* ========================================================================
 * MXFP4 weight GEMM.  The pages name low-bit weight GEMMs as the largest
 * mixed-precision win ("5分钟上手TileLang", section "H100 实测": WFP4 mixed
 * precision; section "进阶方向": dequantize_gemm with W4A8 and MXFP4;
 * "TileLang：让GPU编程像Python一样简单的高性能计算新范式": WINT2AFP16) but
 * define no format.  Reading taken: B is stored in the OCP Microscaling
 * MXFP4 format and dequantised to fp16 before an fp16 GEMM:
 *
 *   code(k, n) = 4-bit FP4 E2M1 element: byte Bq[n*ldbq + k/2], low nibble
 *                for even k, high nibble for odd k (B is stored in the
 *                [out][in] orientation of a linear layer's weight: each
 *                column's k run is contiguous, so a 32-element MX block is 16
 *                bytes);
 *   X(k, n)    = 8-bit E8M0 scale shared by the 32 k of a block:
 *                S[(k/32)*lds + n] (block-major, n contiguous);
 *   Bdeq[k][n] = fp16_rne( e2m1(code) * 2^(X - 127) )   (X = 255: NaN)
 *   C          = the fp16 GEMM of A and Bdeq (oracle_gemm_ex, in_fmt 0).
 *
 * E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa; exponent
 * 0 is subnormal (0 or 0.5); no infinities or NaNs.  E8M0: an unsigned
 * power-of-two exponent with bias 127, 255 encoding NaN.
 * ======================================================================== */

double oracle_f64_from_e2m1(uint8_t code)
{
    const int s = (code >> 3) & 1;
    const int e = (code >> 1) & 3;
    const int m = code & 1;
    double mag = (e == 0) ? ldexp((double)m, -1) : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

double oracle_f64_from_e8m0(uint8_t x)
{
    if (x == 255) return NAN;
    return ldexp(1.0, (int)x - 127);
}

/* Bdeq (K×N fp16 bits, row stride ldb) from the packed codes (N rows of
 * ldbq bytes) and scales.  Returns 0, or -1 on bad arguments. */
int oracle_mxfp4_dequant_f16(const uint8_t* Bq, int64_t ldbq, const uint8_t* S, int64_t lds,
                             int64_t K, int64_t N, uint16_t* Bdeq, int64_t ldb)
{
    if (K < 0 || N < 0 || ldbq < (K + 1) / 2 || lds < N || ldb < N) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t n = 0; n < N; ++n) {
            uint8_t byte = Bq[n * ldbq + k / 2];
            uint8_t code = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            double v = oracle_f64_from_e2m1(code) * oracle_f64_from_e8m0(S[(k / 32) * lds + n]);
            Bdeq[k * ldb + n] = oracle_f16_from_f64(v);
        }
    }
    return 0;
}

/* ========================================================================
 * 2:4 structured-sparse A.  The pages name a sparse GEMM on 2:4 sparse tensor
 * cores ("TileLang：让GPU编程像Python一样简单的高性能计算新范式", T.gemm_sp(A_sparse,
 * B, C)) without fixing a storage format.  Reading taken: A (M×K, K a
 * multiple of 32) has at most two nonzeros in every aligned group of four
 * consecutive k; it is stored as
 *   Ac[i][2*G + h]   the h-th kept value (h = 0, 1; increasing k) of group G
 *                    (G = k/4), fp16, row stride ldac (>= K/2);
 *   E[i][w]          32-bit metadata word w (row stride lde >= K/32 words):
 *                    group G = 8w + g sits in bits 4g .. 4g+3, low two bits
 *                    = position (0..3) of the first kept value, high two bits
 *                    = position of the second, first < second.
 * Dense A: A[i][4G + pos_h] = Ac[i][2G + h], every other element +0.
 * C is then the GEMM of the dense A and B (oracle_gemm_ex with fp16 or bf16
 * inputs).
 * ======================================================================== */

/* Dense A (M×K 16-bit patterns, row stride lda) from Ac and E.  Returns 0, -1
 * on bad sizes, -2 if any group's positions are not first < second. */
int oracle_sp24_decompress(const uint16_t* Ac, int64_t ldac, const uint32_t* E, int64_t lde,
                           int64_t M, int64_t K, uint16_t* A, int64_t lda)
{
    if (M < 0 || K < 0 || (K % 32) != 0 || ldac < K / 2 || lde < K / 32 || lda < K) return -1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t k = 0; k < K; ++k) A[i * lda + k] = 0;  /* +0 in fp16 and bf16 */
        for (int64_t G = 0; G < K / 4; ++G) {
            uint32_t word = E[i * lde + G / 8];
            uint32_t nib = (word >> (4 * (G % 8))) & 15u;
            uint32_t p0 = nib & 3u, p1 = (nib >> 2) & 3u;
            if (p0 >= p1) return -2;
            A[i * lda + 4 * G + p0] = Ac[i * ldac + 2 * G];
            A[i * lda + 4 * G + p1] = Ac[i * ldac + 2 * G + 1];
        }
    }
    return 0;
}
