// The element-wise epilogue of the pair and one-CTA kernels, for one
// 64-column chunk of one accumulator row held by one thread:
//
//   x[t] = act( acc[t] + bias[col0 + t] ) + R[row][col0 + t]      (fp32)
//   C[row][col0 + t] = out(x[t])                                   (one rounding)
//
// This is the ReLU epilogue of the pages (an element-wise step on the fp32
// accumulator before the final copy: "TileLang：让GPU编程像Python一样简单的高性能
// 计算新范式", the T.Parallel loop over C_local) extended with an optional
// per-column bias, an optional residual matrix and an optional fp32 output.
// The 32 threads of a warp hold 32 consecutive rows; the chunk is staged in
// 128-byte-swizzled shared memory and written with TMA stores (clipped at the
// M and N edges).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace tg {

// Epilogue arguments shared by the tile kernels (part of PersistentParams).
struct EpilogueArgs {
    const float* bias = nullptr;   // N values, or null
    const void* resid = nullptr;   // M×N of the input element type (row stride ldr), or null
    int64_t ldr = 0;
    int32_t bias_vec = 0;          // bias is 16-byte aligned: vector loads
    int32_t resid_vec = 0;         // resid and ldr allow 16-byte row loads
};

// The whole epilogue as the host plans it.
struct EpilogueSpec {
    int32_t relu = 0;
    EpilogueArgs e;
    int32_t out_f32 = 0;  // C is fp32 instead of the input type
};

template <typename T>
__device__ __forceinline__ void load8_to_float(const T* src, float (&out)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = Elem16<T>::to_float(e[i]);
}

// x (64 accumulator values of row `row`, columns col0..col0+63) → final fp32
// values, before the output rounding.
template <typename T>
__device__ __forceinline__ void epilogue_math(float (&x)[64], const EpilogueArgs& e, int relu,
                                              int row, int col0, int M, int N) {
    const bool full = col0 + 64 <= N;
    if (e.bias != nullptr) {
        if (e.bias_vec && full) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const float4 b = __ldg(reinterpret_cast<const float4*>(e.bias + col0) + t);
                x[4 * t] += b.x;
                x[4 * t + 1] += b.y;
                x[4 * t + 2] += b.z;
                x[4 * t + 3] += b.w;
            }
        } else {
#pragma unroll
            for (int t = 0; t < 64; ++t)
                if (col0 + t < N) x[t] += __ldg(e.bias + col0 + t);
        }
    }
    if (relu) {
#pragma unroll
        for (int t = 0; t < 64; ++t) x[t] = relu_f32(x[t]);
    }
    if (e.resid != nullptr && row < M) {
        const T* rp = static_cast<const T*>(e.resid) + static_cast<int64_t>(row) * e.ldr + col0;
        if (e.resid_vec && full) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                float r[8];
                load8_to_float(rp + 8 * t, r);
#pragma unroll
                for (int i = 0; i < 8; ++i) x[8 * t + i] += r[i];
            }
        } else {
#pragma unroll
            for (int t = 0; t < 64; ++t)
                if (col0 + t < N) x[t] += Elem16<T>::to_float(rp[t]);
        }
    }
}

// Stage and store one chunk of 64 columns already rounded to the 16-bit type
// (h[t] holds columns 2t and 2t + 1, the first in the low half).  cbuf: this
// warp's two 4 KB staging buffers; buf: which one is used next (toggled).
__device__ __forceinline__ void epilogue_store_packed(const uint32_t (&h)[32], uint32_t cbuf,
                                                      int& buf, const void* tmC, uint64_t policy,
                                                      int row0, int col0, int M, int N, int lane) {
    if (lane == 0) bulk_wait_group_read<1>();  // the buffer used two chunks ago is free
    __syncwarp();
    const uint32_t cb = cbuf + static_cast<uint32_t>(buf) * 4096u;
    const uint32_t row_addr = cb + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        st_shared_v4(row_addr + ((static_cast<uint32_t>(c) ^ (lane & 7u)) << 4), h[4 * c],
                     h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (row0 < M && col0 < N) tma_store_2d_hint(tmC, cb, col0, row0, policy);
        bulk_commit_group();
    }
    buf ^= 1;
}

// Stage and store one chunk.  cbuf: this warp's two 4 KB staging buffers;
// buf: which one the 16-bit path uses next (toggled).  row0: the warp's first
// row (stores are clipped at M and N by the tensor map).  out_f32 (uniform
// over the grid): C is fp32, its tensor map has 32×32 boxes.
template <typename T>
__device__ __forceinline__ void epilogue_store(const float (&x)[64], uint32_t cbuf, int& buf,
                                               const void* tmC, uint64_t policy, int row0,
                                               int col0, int M, int N, int lane, bool out_f32) {
    if (!out_f32) {
        uint32_t h[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) h[t] = Elem16<T>::pack2(x[2 * t], x[2 * t + 1]);
        epilogue_store_packed(h, cbuf, buf, tmC, policy, row0, col0, M, N, lane);
    } else {
        // fp32: 256 bytes per row, two 32-column boxes, one per buffer.
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint32_t row_addr = cbuf + static_cast<uint32_t>(half) * 4096u +
                                      static_cast<uint32_t>(lane) * 128u;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float* q = x + 32 * half + 4 * c;
                st_shared_v4(row_addr + ((static_cast<uint32_t>(c) ^ (lane & 7u)) << 4),
                             __float_as_uint(q[0]), __float_as_uint(q[1]), __float_as_uint(q[2]),
                             __float_as_uint(q[3]));
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (row0 < M && col0 < N) tma_store_2d_hint(tmC, cbuf, col0, row0, policy);
            if (row0 < M && col0 + 32 < N) tma_store_2d_hint(tmC, cbuf + 4096u, col0 + 32, row0, policy);
            bulk_commit_group();
        }
    }
}

}  // namespace tg
