// MXFP4 weight decoding for sm_103a.
//
// The pages name low-bit weight GEMMs (WFP4, W4A8, MXFP4 in dequantize_gemm:
// "5分钟上手TileLang", sections "H100 实测" and "进阶方向") without defining a
// format.  The format read here is the OCP Microscaling MXFP4 encoding:
//   element  FP4 E2M1, 4 bits: sign, 2 exponent bits (bias 1), 1 mantissa
//            bit; exponent 0 is subnormal (0 or 0.5); values up to ±6;
//   scale    E8M0, 8 bits: 2^(X - 127), X = 255 is NaN; one scale per 32
//            consecutive k of a column.
// Storage: B's codes are N rows (one per column of B, the [out][in]
// orientation of a linear layer's weight) of ceil(K/2) bytes, two elements
// per byte along k (low nibble = even k), row stride ldbq bytes; scales are
// ceil(K/32)×N bytes (block-major, n contiguous), row stride lds.  The
// decoded weight is the fp16 number
//   Bdeq[k][n] = fp16_rne( e2m1(code) × 2^(X - 127) ).
//
// Fast path: cvt.rn.f16x2.e2m1x2 turns a byte (two codes) into two exact fp16
// values; one mul.rn.f16x2 by the fp16 number 2^(X - 127) then rounds the
// exact product once, which is Bdeq.  That factor is an fp16 number for
// 103 ≤ X ≤ 142 (subnormal below X = 113); for X ≤ 99 every product is below
// half the smallest fp16 subnormal, so a factor of +0 gives the correct ±0.
// Other scales (100..102, 143..255) take an fp32 route that is exact for
// every X (the fp32 product of an E2M1 value and 2^(X-127) is exact, then one
// fp32 → fp16 rounding).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"

namespace tg {

// Shared-memory accesses of the converter warps (32-bit shared addresses).
__device__ __forceinline__ uint4 mx_ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t mx_ld_shared_u8(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t mx_ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void mx_st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b));
}

// tcgen05.mma with the A operand in tensor memory (K-major: lane = row,
// 32-bit column = two consecutive k, lower k in the low half), B in shared
// memory.
__device__ __forceinline__ void mx_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The eight MMAs of one 128-k MXFP4 unit and its two release commits, issued
// by one elected lane of a converged warp in one block: D (+)= W · Xᵀ with
// the decoded weights W (128 n × 16 k per MMA) at tensor-memory columns
// a_tmem + 8 k and the activation tile X in shared memory, its descriptor
// b_desc advanced 32 bytes per 16 k inside a 64-k box and BOX16 (the box
// size in 16-byte units) from one box to the next.  first != 0: the first
// MMA overwrites D.  Fewer instructions per unit on the issuing warp, which
// shares its scheduler with the decoding warps.
template <uint32_t BOX16>
__device__ __forceinline__ void mx_unit_mma_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t first, uint32_t bar_op,
                                                  uint32_t bar_a) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 a;\n\t.reg .b64 b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.eq.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "add.u32 a, %1, 8;\n\tadd.u64 b, %2, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
        "add.u32 a, %1, 16;\n\tadd.u64 b, %2, 4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
        "add.u32 a, %1, 24;\n\tadd.u64 b, %2, 6;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
        "add.u32 a, %1, 32;\n\tadd.u64 b, %2, %7;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
        "add.u32 a, %1, 40;\n\tadd.u64 b, b, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
        "add.u32 a, %1, 48;\n\tadd.u64 b, b, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
        "add.u32 a, %1, 56;\n\tadd.u64 b, b, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t"
        "}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(first), "r"(bar_op), "r"(bar_a),
        "n"(BOX16)
        : "memory");
}

// This warp's 32 lanes (its lane quarter) × 32 consecutive 32-bit columns.
__device__ __forceinline__ void mx_tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void mx_tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ bool mx_fast_scale(uint32_t X) {
    return X <= 99u || (X >= 103u && X <= 142u);
}

// fp16 bits of the fast-path factor for scale byte X (mx_fast_scale(X)).
__device__ __forceinline__ uint32_t mx_factor_bits(uint32_t X) {
    if (X <= 99u) return 0u;                      // products underflow to ±0
    if (X <= 112u) return 1u << (X - 103u);       // subnormal: 2^-24 · 2^(X-103)
    return (X - 112u) << 10;                      // normal: biased exponent X - 127 + 15
}

// Eight codes (one 32-bit word: byte p holds elements 2p (low nibble) and
// 2p+1) → eight fp16 values, scaled by the factor pairs f[p] (fp16x2: element
// 2p in the low half).
__device__ __forceinline__ uint4 mx_decode8_fast(uint32_t w, const uint32_t (&f)[4]) {
    uint32_t h0, h1, h2, h3;
    asm("{\n\t"
        ".reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t"
        "}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
    uint4 o;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o.x) : "r"(h0), "r"(f[0]));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o.y) : "r"(h1), "r"(f[1]));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o.z) : "r"(h2), "r"(f[2]));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o.w) : "r"(h3), "r"(f[3]));
    return o;
}

// One code with scale byte X, exact for every X (fp16 bits).
__device__ __forceinline__ uint16_t mx_decode1_exact(uint32_t code, uint32_t X) {
    const uint32_t e = (code >> 1) & 3u;
    const uint32_t m = code & 1u;
    const float mag = e == 0u ? 0.5f * static_cast<float>(m)
                              : (1.0f + 0.5f * static_cast<float>(m)) *
                                    static_cast<float>(1u << (e - 1u));
    float s;
    if (X == 255u)
        s = __uint_as_float(0x7fc00000u);  // NaN scale
    else if (X == 0u)
        s = __uint_as_float(0x00400000u);  // 2^-127, an fp32 subnormal
    else
        s = __uint_as_float(X << 23);      // 2^(X-127)
    float v = mag * s;                     // exact (or ±inf / NaN where fp16 is too)
    if (code & 8u) v = -v;
    return __half_as_ushort(__float2half_rn(v));
}

// Eight codes with per-element scale bytes x[0..7], exact for every scale.
__device__ __forceinline__ uint4 mx_decode8_exact(uint32_t w, const uint32_t (&x)[8]) {
    uint32_t h[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t lo = mx_decode1_exact((w >> (8 * p)) & 15u, x[2 * p]);
        const uint32_t hi = mx_decode1_exact((w >> (8 * p + 4)) & 15u, x[2 * p + 1]);
        h[p] = lo | (hi << 16);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

// Bdeq as a K×N fp16 matrix (row stride ldo elements, a multiple of 8; 16-byte
// aligned base) from the packed codes and scales: a transpose through shared
// memory, one 64 k × 64 n tile per block iteration.  Codes rows and scale rows
// are 16-byte aligned (ldbq, lds multiples of 16).  256 threads.
__global__ void __launch_bounds__(256)
    tg_mxfp4_dequant_f16(const uint8_t* __restrict__ Bq, int64_t ldbq,
                         const uint8_t* __restrict__ S, int64_t lds, int64_t K, int64_t N,
                         uint16_t* __restrict__ out, int64_t ldo) {
    __shared__ __align__(16) uint16_t tile[64][64 + 8];  // [k][n]
    const int64_t tiles_n = (N + 63) / 64;
    const int64_t tiles = tiles_n * ((K + 63) / 64);
    const int nl = threadIdx.x >> 2;  // decode: column n0 + nl, codes k0 + 16 kq .. + 15
    const int kq = threadIdx.x & 3;
    grid_dependency_wait();  // (a plain launch: returns at once)
    grid_launch_dependents();  // the GEMM on the decoded weights may set up meanwhile
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t n0 = (t % tiles_n) * 64;
        const int64_t k0 = (t / tiles_n) * 64;
        const int64_t n = n0 + nl;
        const int64_t kb = k0 + 16 * kq;
        uint32_t h[8];  // 16 fp16, k ascending, two per word
        if (n < N && kb + 16 <= K) {
            const uint2 wv = *reinterpret_cast<const uint2*>(Bq + n * ldbq + kb / 2);
            const uint32_t X = S[(kb / 32) * lds + n];  // 16 aligned k: one block
            uint4 lo, hi;
            if (mx_fast_scale(X)) {
                const uint32_t f = mx_factor_bits(X) * 0x10001u;
                const uint32_t fj[4] = {f, f, f, f};
                lo = mx_decode8_fast(wv.x, fj);
                hi = mx_decode8_fast(wv.y, fj);
            } else {
                const uint32_t x[8] = {X, X, X, X, X, X, X, X};
                lo = mx_decode8_exact(wv.x, x);
                hi = mx_decode8_exact(wv.y, x);
            }
            h[0] = lo.x; h[1] = lo.y; h[2] = lo.z; h[3] = lo.w;
            h[4] = hi.x; h[5] = hi.y; h[6] = hi.z; h[7] = hi.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t pair = 0;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int64_t k = kb + 2 * j + e;
                    if (n < N && k < K) {
                        const uint32_t byte = Bq[n * ldbq + k / 2];
                        const uint32_t code = (k & 1) ? (byte >> 4) : (byte & 15u);
                        pair |= static_cast<uint32_t>(mx_decode1_exact(code, S[(k / 32) * lds + n]))
                                << (16 * e);
                    }
                }
                h[j] = pair;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            tile[16 * kq + 2 * j][nl] = static_cast<uint16_t>(h[j] & 0xFFFFu);
            tile[16 * kq + 2 * j + 1][nl] = static_cast<uint16_t>(h[j] >> 16);
        }
        __syncthreads();
        // write out: row k0 + (tid / 4), columns n0 + 16 (tid % 4) .. + 15
        const int r = threadIdx.x >> 2;
        const int c0 = 16 * (threadIdx.x & 3);
        const int64_t k = k0 + r;
        if (k < K) {
            uint16_t* dst = out + k * ldo + n0 + c0;
            if (n0 + c0 + 16 <= N) {
                const uint4* srow = reinterpret_cast<const uint4*>(&tile[r][c0]);
                reinterpret_cast<uint4*>(dst)[0] = srow[0];
                reinterpret_cast<uint4*>(dst)[1] = srow[1];
            } else {
                for (int c = 0; c < 16 && n0 + c0 + c < N; ++c) dst[c] = tile[r][c0 + c];
            }
        }
        __syncthreads();
    }
}

}  // namespace tg
