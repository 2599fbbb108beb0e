// Persistent, warp-specialised FP16 GEMM for sm_103a:  C = epi(A · B).
//
// A: M×K row-major (K contiguous)  -> K-major tensor-core operand.
// B: K×N row-major (N contiguous)  -> MN-major tensor-core operand.
// C: M×N row-major fp16.
//
// One CTA per SM walks output tiles of 128×BN (tile_coord order).  Roles:
//   warp 0      producer: TMA loads of a 128×64 A box and BN/64 64×64 B boxes
//               per k step into a STAGES-deep shared-memory ring, signalled on
//               full[s] as transaction bytes; waits on empty[s] before reuse.
//   warp 1      MMA issuer: allocates 2×BN TMEM columns (two fp32
//               accumulators), issues four 128×BN×16 tcgen05.mma per k step,
//               releases ring slots with tcgen05.commit -> empty[s] and hands a
//               finished accumulator to the epilogue via tmem_full[a].
//   warps 2..5  epilogue: tcgen05.ld of 32 rows each (TMEM lane quarter =
//               warp % 4), bias / ReLU / residual on the fp32 value, round
//               to the output type, stage in a 128-byte-swizzled shared
//               buffer, TMA store (epilogue.cuh); tmem_empty[a]
//               returns the accumulator to the MMA warp, so the epilogue of
//               tile t overlaps the main loop of tile t+1.
//
// The structure follows the generated Hopper kernel shown in "TileLang：比
// Triton 低一层的 tile 语言" (section "它生成了什么": TMA descriptors, a ring of
// "data arrived" / "buffer empty" mbarriers, producer and consumer warps),
// re-designed for tcgen05: the accumulator lives in TMEM instead of
// registers, so the epilogue runs in its own warps and the register
// hand-over between warpgroups of that design is not needed.
#pragma once

#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "sm103_ptx.cuh"
#include "tile_schedule.h"

namespace tg {

// Set (OR of 1 << role) by any kernel that gave up on a wait; read and
// cleared by tg_sync_status().
__device__ unsigned int g_wait_timeout_flags;

struct PersistentParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n, num_tiles, k_blocks;
    int32_t group_m;
    int32_t relu;
    int32_t inject;  // 1: withhold the first tmem_full signal (fault-path test)
    uint64_t timeout_ns;
    EpilogueArgs e;       // bias / residual (null: none)
    int32_t out_f32 = 0;  // 1: C is fp32 (tensor map with 32×32 boxes)
    // Pair kernel only: k-pieces and column halves per tail tile
    // (tile_schedule.h), and for split > 1 the partial slots (one per
    // cluster) and the tail tiles' counters (eight per tile, zero between
    // launches).
    int32_t split = 1;
    int32_t split_n = 1;
    float* ws = nullptr;
    uint32_t* counters = nullptr;
};

enum : unsigned int { kRoleProducer = 1u, kRoleMma = 2u, kRoleEpilogue = 4u, kRoleDrain = 8u };

template <int BN, int STAGES>
struct PersistentCfg {
    static constexpr int BM = 128;
    static constexpr int BK = 64;
    static constexpr int kThreads = 192;
    static constexpr uint32_t kABytes = BM * BK * 2;              // 16 KB
    static constexpr uint32_t kBBytes = BN * BK * 2;              // BN/64 boxes of 8 KB
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kCBuf = 32 * 64 * 2;                // 32 rows × 64 cols fp16
    static constexpr uint32_t kCBytes = 4 * 2 * kCBuf;            // 4 warps × 2 buffers
    static constexpr uint32_t kBarBytes = 256;
    static constexpr uint32_t kTmemCols = 2 * BN;                 // two fp32 accumulators
    static constexpr uint32_t kSmemBytes =
        1024 /*alignment slack*/ + STAGES * kStageBytes + kCBytes + kBarBytes;
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64..256, multiple of 64");
    static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols >= 32 && kTmemCols <= 512,
                  "TMEM columns must be a power of two in [32, 512]");
};

// EX = false: the plain epilogue only (no bias, no residual, 16-bit C); the
// other epilogue paths are compiled out, which keeps the kernel's code small
// for the latency-bound launches of small problems.
template <int BN, int STAGES, typename T = __half, bool EX = true>
__global__ void __launch_bounds__(192, 1)
    tg_gemm_f16_persistent(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC, const PersistentParams p) {
    using Cfg = PersistentCfg<BN, STAGES>;
    constexpr int BM = Cfg::BM;
    constexpr int BK = Cfg::BK;
    constexpr uint32_t kABytes = Cfg::kABytes;
    constexpr uint32_t kBBytes = Cfg::kBBytes;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base;
    const uint32_t sB = sA + STAGES * kABytes;
    const uint32_t sC = sB + STAGES * kBBytes;
    const uint32_t sBar = sC + Cfg::kCBytes;
    // barrier slots (8 bytes each)
    const uint32_t bar_full = sBar;                      // [STAGES]
    const uint32_t bar_empty = sBar + 8 * STAGES;        // [STAGES]
    const uint32_t bar_tfull = sBar + 16 * STAGES;       // [2]
    const uint32_t bar_tempty = bar_tfull + 16;          // [2]
    const uint32_t bar_drain = bar_tempty + 16;          // [1]
    const uint32_t slot_tmem = bar_drain + 8;            // u32: TMEM base address
    uint32_t* const tmem_slot_ptr = reinterpret_cast<uint32_t*>(base_ptr + (slot_tmem - base));
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot_ptr + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + 8 * a, 1);
            mbar_init(bar_tempty + 8 * a, 4);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(slot_tmem, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot_ptr;
    // Producer set-up that reads no data of the previous kernel (its cache
    // policy, its first tile's block coordinates) is done before the
    // dependency wait, with the first ring's worth of this CTA's operand
    // tiles prefetched into L2 while the previous kernel finishes.
    uint64_t a_policy = 0;
    TileCoord tc_first{0, 0};
    if (warp == 0 && lane == 0) {
        a_policy = policy_evict_last();
        if (static_cast<int>(blockIdx.x) < p.num_tiles) {
            tc_first = tile_coord(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m);
            for (int kb = 0; kb < STAGES && kb < p.k_blocks; ++kb) {
                tma_prefetch_2d(&tmA, kb * BK, tc_first.m_blk * BM);
#pragma unroll
                for (int j = 0; j < BN / 64; ++j)
                    tma_prefetch_2d(&tmB, tc_first.n_blk * BN + 64 * j, kb * BK);
            }
        }
    }
    grid_dependency_wait();  // the previous kernel's writes are visible from here on
    grid_launch_dependents();

    auto fail = [&](unsigned int role) {
        atomicOr(&g_wait_timeout_flags, role);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;  // last load per stage
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                const TileCoord tc = tile == static_cast<int>(blockIdx.x)
                                         ? tc_first
                                         : tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m);
                const int m0 = tc.m_blk * BM;
                const int n0 = tc.n_blk * BN;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.timeout_ns, abort_flag)) {
                        fail(kRoleProducer);
                        ok = false;
                        break;
                    }
                    const uint32_t full = bar_full + 8 * stage;
                    mbar_arrive_expect_tx(full, Cfg::kStageBytes);
                    // A panels are reread by every column block of the raster
                    // group: kept in L2 ahead of B and C
                    tma_load_2d_hint(sA + stage * kABytes, &tmA, full, kb * BK, m0, a_policy);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(sB + stage * kBBytes + j * 8192, &tmB, full, n0 + 64 * j,
                                    kb * BK);
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Drain: every load this thread issued must have landed before the
            // CTA may exit (normally already true).
            for (int s = 0; s < STAGES; ++s)
                if (issued_mask & (1u << s))
                    if (!mbar_wait(bar_full + 8 * s, (issued_parity >> s) & 1u, p.timeout_ns,
                                   nullptr))
                        atomicOr(&g_wait_timeout_flags, kRoleDrain);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (warp-uniform control flow and
        // operands); one elected lane issues each stage's MMAs and commit.
        // A wait counts as met only if every lane saw it met.
        {
            static_assert(BK == 64, "stage4_mma_ss_elect issues 64 k per stage");
            constexpr uint32_t idesc =
                idesc_f16_f32(BM, BN, /*a_mn=*/false, /*b_mn=*/true, Elem16<T>::kFmt);
            auto warp_wait = [&](uint32_t bar, uint32_t parity, const volatile int* ab) {
                const bool r = mbar_wait(bar, parity, p.timeout_ns, ab);
                return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
            };
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!warp_wait(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag)) {
                    if (lane == 0) fail(kRoleMma);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!warp_wait(bar_full + 8 * stage, phase, abort_flag)) {
                        if (lane == 0) fail(kRoleMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    // A: K-major, +32 B per 16-element k slice inside the 128 B row.
                    // B: MN-major, 16 k-rows of 128 B per slice; 64-wide N chunks 8 KB apart.
                    stage4_mma_ss_elect<2, 128>(
                        d_tmem, smem_desc_sw128(sA + stage * kABytes, 16, 1024),
                        smem_desc_sw128(sB + stage * kBBytes, 8192, 1024), idesc,
                        kb == 0 ? 1u : 0u, bar_empty + 8 * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (!(p.inject == 1 && it == 0)) {
                    __syncwarp();
                    if (lane == 0) mma_commit(bar_tfull + 8 * acc);
                }
            }
            // Drain: all MMAs issued by this warp complete before TMEM is freed.
            __syncwarp();
            if (lane == 0) mma_commit(bar_drain);
            if (!warp_wait(bar_drain, 0, nullptr) && lane == 0)
                atomicOr(&g_wait_timeout_flags, kRoleDrain);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t cbuf = sC + static_cast<uint32_t>((warp - 2) * 2) * Cfg::kCBuf;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        const uint64_t c_policy = policy_evict_first();  // C is written once, never reread
        int buf = 0;
        int it = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const TileCoord tc = tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m);
            const int m0 = tc.m_blk * BM;
            const int n0 = tc.n_blk * BN;
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            int ok = 1;
            if (lane == 0)
                ok = mbar_wait(bar_tfull + 8 * acc, acc_phase, p.timeout_ns, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) fail(kRoleEpilogue);
                break;
            }
            tc_fence_after_sync();
            const int row0 = m0 + 32 * q;
#pragma unroll 1
            for (int j = 0; j < BN / 64; ++j) {
                uint32_t v0[32], v1[32];
                const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(acc * BN + j * 64);
                tmem_ld_x32(taddr, v0);
                tmem_ld_x32(taddr + 32, v1);
                if (j == BN / 64 - 1) {
                    // accumulator fully read: hand it back to the MMA warp
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
                }
                float x[64];
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    x[t] = __uint_as_float(v0[t]);
                    x[32 + t] = __uint_as_float(v1[t]);
                }
                epilogue_math<T>(x, EX ? p.e : EpilogueArgs{}, p.relu, row0 + lane, n0 + 64 * j,
                                 p.M, p.N);
                epilogue_store<T>(x, cbuf, buf, &tmC, c_policy, row0, n0 + 64 * j, p.M, p.N, lane,
                                  EX && p.out_f32 != 0);
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

// K == 0: C = epi(0) = +0 over the M×N region (row stride ldc).
__global__ void tg_fill_zero_f16(__half* C, int64_t M, int64_t N, int64_t ldc) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / N, c = i - r * N;
        C[r * ldc + c] = __ushort_as_half(0);
    }
}

// K == 0 with a bias, a residual or an fp32 output: the product is the empty
// sum (+0), so C = out(act(+0 + bias[j]) + R[i][j]) element by element.
template <typename T>
__global__ void tg_epilogue_only(void* C, int64_t ldc, int32_t out_f32, EpilogueArgs e,
                                 int32_t relu, int64_t M, int64_t N) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / N, c = i - r * N;
        float v = 0.0f;
        if (e.bias != nullptr) v += e.bias[c];
        if (relu) v = relu_f32(v);
        if (e.resid != nullptr)
            v += Elem16<T>::to_float(static_cast<const T*>(e.resid)[r * e.ldr + c]);
        if (out_f32)
            static_cast<float*>(C)[r * ldc + c] = v;
        else
            static_cast<T*>(C)[r * ldc + c] = Elem16<T>::from_float(v);
    }
}

}  // namespace tg
