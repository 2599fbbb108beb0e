// Staging copy for layouts the tensor memory-access unit cannot address.
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace tg {

// Copy a rows×cols matrix of E (2- or 4-byte elements) between two row
// strides, any alignment (used to stage an operand whose layout the tensor
// memory-access unit cannot address into an aligned buffer, and a result back
// out of one).  A warp takes 256 consecutive elements of one row per step,
// lane l elements l, l + 32, ..., l + 224: every load and store instruction
// of the warp touches 32 consecutive elements.  (With 8 consecutive elements
// per thread each instruction spanned 512 bytes at a 16-byte lane stride, and
// copying the 8192×4096 fp16 A of the MLP shape took 70 us.)
template <typename E>
__global__ void tg_copy_matrix(const E* __restrict__ src, int64_t ld_src, E* __restrict__ dst,
                               int64_t ld_dst, int64_t rows, int64_t cols) {
    constexpr int kPerLane = 8;
    constexpr int64_t kSeg = 32 * kPerLane;  // elements per warp step
    const int lane = threadIdx.x & 31;
    const int64_t segs = (cols + kSeg - 1) / kSeg;
    const int64_t total = rows * segs;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    grid_dependency_wait();  // (a plain launch: returns at once)
    grid_launch_dependents();  // the next kernel may set up while this one copies
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         w < total; w += nwarps) {
        const int64_t r = w / segs;
        const int64_t c0 = (w - r * segs) * kSeg;
        const E* s = src + r * ld_src + c0;
        E* d = dst + r * ld_dst + c0;
        const int64_t n = cols - c0 < kSeg ? cols - c0 : kSeg;
        E v[kPerLane];
#pragma unroll
        for (int j = 0; j < kPerLane; ++j)
            if (lane + 32 * j < n) v[j] = s[lane + 32 * j];
#pragma unroll
        for (int j = 0; j < kPerLane; ++j)
            if (lane + 32 * j < n) d[lane + 32 * j] = v[j];
    }
}

}  // namespace tg
