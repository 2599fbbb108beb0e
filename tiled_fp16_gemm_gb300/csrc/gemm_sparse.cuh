// 2:4 structured-sparse GEMM for sm_103a:  C = epi(A · B) with A sparse.
//
// A (M×K) keeps two values in every aligned group of four k.  It is stored
// compressed (Ac: M × K/2, the kept values in increasing k) with metadata E
// (M × K/32 32-bit words: group g of word w — k = 32 w + 4 g .. + 3 — in bits
// 4g .. 4g+3, low two bits the first kept position, high two the second).
// The pages name the operation (T.gemm_sp on 2:4 sparse tensor cores:
// "TileLang：让GPU编程像Python一样简单的高性能计算新范式", section on sparse
// computation); this kernel runs it on tcgen05.mma.sp, which consumes the
// compressed A tile as the operand and multiplies it against 32 k of B per
// instruction (twice the k of a dense kind::f16 MMA).
//
// Persistent CTAs walk 128×128 output tiles (tile_coord order).  Roles:
//   warp 0      producer: per 128-k stage one TMA box of Ac (128 rows × 64
//               values), two of B (64 n × 128 k each) and one of E (128 rows ×
//               4 words) into a 3-deep ring;
//   warp 1      MMA: four tcgen05.mma.sp (128 × 128 × 32) per stage into one of
//               two fp32 accumulators in tensor memory;
//   warps 2..5  epilogue (epilogue.cuh), overlapped with the next tile;
//   warps 6..9  metadata: tensor memory holds the sparse metadata of one MMA in
//               one 32-bit column whose lanes interleave rows — within each
//               16-row block, lane l's low (high) 16 bits hold the metadata of
//               row l & 7 (row 8 + (l & 7)) for the k half l >> 3 of the 32 k.
//               Warp w rewrites its lane quarter's words from the E tile with
//               one tcgen05.st per stage (rows past M and words past K/32 get
//               a valid pattern; their values are zero-filled).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "gemm_persistent.cuh"
#include "sm103_ptx.cuh"
#include "tile_schedule.h"

namespace tg {

constexpr unsigned int kRoleMeta = 32u;

struct SparseCfg {
    static constexpr int BM = 128;
    static constexpr int BN = 128;
    static constexpr int BK = 128;      // dense-equivalent k per stage
    static constexpr int STAGES = 3;
    static constexpr int kThreads = 320;
    static constexpr uint32_t kABytes = BM * (BK / 2) * 2;  // 16 KB of kept values
    static constexpr uint32_t kBBytes = BK * BN * 2;        // 32 KB: two 64-column boxes
    static constexpr uint32_t kEBytes = BM * (BK / 32) * 4; // 2 KB of metadata
    static constexpr uint32_t kStageBytes = kABytes + kBBytes + kEBytes;
    static constexpr uint32_t kCBuf = 32 * 64 * 2;
    static constexpr uint32_t kCBytes = 4 * 2 * kCBuf;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kMetaCol0 = 2 * BN;           // after the two accumulators
    // Each MMA's metadata column sits on a 16-column boundary: stage s, k
    // slice k at kMetaCol0 + 64 s + 16 k.
    static constexpr uint32_t kMetaStageCols = 64;
    static constexpr uint32_t kMetaSliceCols = 16;
    static constexpr uint32_t kSmemBytes =
        1024 + STAGES * (kABytes + kBBytes) + STAGES * kEBytes + kCBytes + 256;
    static_assert(kMetaCol0 + kMetaStageCols * STAGES <= kTmemCols,
                  "metadata columns exceed tensor memory");
};

struct SparseParams {
    PersistentParams base;  // M, N, K, tiles, group, epilogue, timeout
    int32_t words;          // K / 32: metadata words per row
};

__device__ __forceinline__ void mma_f16_sp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t meta_tmem, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.sp.cta_group::1.kind::f16 [%0], %1, %2, [%3], %4, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(meta_tmem), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One stage (128 dense-equivalent k) of the one-CTA sparse kernel: four
// sparse MMAs of 128 × 128 × 32 and the stage's release commit, issued by one
// elected lane of a converged warp in one block.  MMA k reads A 32 B further
// (ad + 2 k), B 4 KB further (bd + 256 k) and metadata 16 columns further.
// first != 0: the first MMA overwrites D.
__device__ __forceinline__ void sp_stage_mma_elect(uint32_t d_tmem, uint64_t ad, uint64_t bd,
                                                   uint32_t meta, uint32_t idesc, uint32_t first,
                                                   uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 m;\n\t.reg .b64 a, b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.eq.b32 p, %5, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "@e tcgen05.mma.sp.cta_group::1.kind::f16 [%0], %1, %2, [%3], %4, p;\n\t"
        "add.u64 a, %1, 2;\n\tadd.u64 b, %2, 256;\n\tadd.u32 m, %3, 16;\n\t"
        "@e tcgen05.mma.sp.cta_group::1.kind::f16 [%0], a, b, [m], %4, t;\n\t"
        "add.u64 a, %1, 4;\n\tadd.u64 b, %2, 512;\n\tadd.u32 m, %3, 32;\n\t"
        "@e tcgen05.mma.sp.cta_group::1.kind::f16 [%0], a, b, [m], %4, t;\n\t"
        "add.u64 a, %1, 6;\n\tadd.u64 b, %2, 768;\n\tadd.u32 m, %3, 48;\n\t"
        "@e tcgen05.mma.sp.cta_group::1.kind::f16 [%0], a, b, [m], %4, t;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t"
        "}" ::"r"(d_tmem),
        "l"(ad), "l"(bd), "r"(meta), "r"(idesc), "r"(first), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t a) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(a)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4_u32(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// EX = false: the plain epilogue only (no bias, no residual, 16-bit C); the
// other epilogue paths are compiled out.
template <typename T, bool EX = true>
__global__ void __launch_bounds__(320, 1)
    tg_gemm_sp24(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmC,
                 const SparseParams sp) {
    using Cfg = SparseCfg;
    constexpr int S = Cfg::STAGES;
    const PersistentParams& p = sp.base;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base;                       // [S] kept values, 128-byte swizzle
    const uint32_t sB = sA + S * Cfg::kABytes;      // [S] B: two 64-column boxes each
    const uint32_t sE = sB + S * Cfg::kBBytes;      // [S] metadata rows of 16 bytes
    const uint32_t sC = sE + S * Cfg::kEBytes;
    const uint32_t sBar = sC + Cfg::kCBytes;
    const uint32_t bar_full = sBar;                 // [S]
    const uint32_t bar_empty = sBar + 8 * S;        // [S]
    const uint32_t bar_meta = sBar + 16 * S;        // [S] metadata in tensor memory
    const uint32_t bar_tfull = sBar + 24 * S;       // [2]
    const uint32_t bar_tempty = bar_tfull + 16;     // [2]
    const uint32_t bar_drain = bar_tempty + 16;
    const uint32_t slot_tmem = bar_drain + 8;
    uint32_t* const tmem_slot_ptr = reinterpret_cast<uint32_t*>(base_ptr + (slot_tmem - base));
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot_ptr + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
            mbar_init(bar_meta + 8 * s, 4);
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
        tma_prefetch_desc(&tmE);
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
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                const TileCoord tc = tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m);
                const int m0 = tc.m_blk * Cfg::BM;
                const int n0 = tc.n_blk * Cfg::BN;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.timeout_ns, abort_flag)) {
                        fail(kRoleProducer);
                        ok = false;
                        break;
                    }
                    const uint32_t full = bar_full + 8 * stage;
                    mbar_arrive_expect_tx(full, Cfg::kStageBytes);
                    tma_load_2d(sA + stage * Cfg::kABytes, &tmA, full, kb * (Cfg::BK / 2), m0);
                    tma_load_2d(sB + stage * Cfg::kBBytes, &tmB, full, n0, kb * Cfg::BK);
                    tma_load_2d(sB + stage * Cfg::kBBytes + Cfg::kBBytes / 2, &tmB, full, n0 + 64,
                                kb * Cfg::BK);
                    tma_load_2d(sE + stage * Cfg::kEBytes, &tmE, full, kb * (Cfg::BK / 32), m0);
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < S; ++s)
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
            // sparse (bit 2), selector 0; A K-major, B MN-major; 128 × 128
            constexpr uint32_t idesc =
                idesc_f16_f32(Cfg::BM, Cfg::BN, /*a_mn=*/false, /*b_mn=*/true,
                              Elem16<T>::kFmt) |
                (1u << 2);
            static_assert(Cfg::BK / 32 == 4 && Cfg::kMetaSliceCols == 16,
                          "sp_stage_mma_elect issues four MMAs 16 metadata columns apart");
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
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::BN);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!warp_wait(bar_full + 8 * stage, phase, abort_flag) ||
                        !warp_wait(bar_meta + 8 * stage, phase, abort_flag)) {
                        if (lane == 0) fail(kRoleMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    // A: 16 kept values (32 B) per 32 k; B: 32 k rows (4 KB) per MMA,
                    // the two 64-column boxes 16 KB apart.
                    sp_stage_mma_elect(
                        d_tmem, smem_desc_sw128(sA + stage * Cfg::kABytes, 16, 1024),
                        smem_desc_sw128(sB + stage * Cfg::kBBytes, 16384, 1024),
                        tmem_base + Cfg::kMetaCol0 +
                            static_cast<uint32_t>(stage) * Cfg::kMetaStageCols,
                        idesc, kb == 0 ? 1u : 0u, bar_empty + 8 * stage);
                    if (++stage == S) {
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
            __syncwarp();
            if (lane == 0) mma_commit(bar_drain);
            if (!warp_wait(bar_drain, 0, nullptr) && lane == 0)
                atomicOr(&g_wait_timeout_flags, kRoleDrain);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const uint32_t cbuf = sC + static_cast<uint32_t>((warp - 2) * 2) * Cfg::kCBuf;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        const uint64_t c_policy = policy_evict_first();
        const EpilogueArgs epi_e = EX ? p.e : EpilogueArgs{};
        int buf = 0;
        int it = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const TileCoord tc = tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m);
            const int row0 = tc.m_blk * Cfg::BM + 32 * q;
            const int n0 = tc.n_blk * Cfg::BN;
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
#pragma unroll 1
            for (int j = 0; j < Cfg::BN / 64; ++j) {
                uint32_t v0[32], v1[32];
                const uint32_t taddr =
                    tmem_base + lane_addr + static_cast<uint32_t>(acc * Cfg::BN + j * 64);
                tmem_ld_x32(taddr, v0);
                tmem_ld_x32(taddr + 32, v1);
                if (j == Cfg::BN / 64 - 1) {
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
                epilogue_math<T>(x, epi_e, p.relu, row0 + lane, n0 + 64 * j, p.M, p.N);
                epilogue_store<T>(x, cbuf, buf, &tmC, c_policy, row0, n0 + 64 * j, p.M, p.N, lane,
                                  EX && p.out_f32 != 0);
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    } else {
        // ------------------------------------------------------------ metadata (warps 6..9)
        // Tensor-memory lane L (quarter q = warp % 4) takes rows r0 = (L & ~15) |
        // (L & 7) and r1 = r0 + 8 of the tile, k half h = (L >> 3) & 1 of each of
        // the stage's four 32-k words.
        const uint32_t L = 32u * static_cast<uint32_t>(warp & 3) + static_cast<uint32_t>(lane);
        const uint32_t r0 = (L & ~15u) | (L & 7u);
        const uint32_t r1 = r0 + 8u;
        const uint32_t h = (L >> 3) & 1u;
        const uint32_t lane_addr = (32u * static_cast<uint32_t>(warp & 3)) << 16;
        constexpr uint32_t kNeutral = 0x4444u;  // positions (0, 1) in every group of a half
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
            const TileCoord tc = tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m);
            const int m0 = tc.m_blk * Cfg::BM;
            const bool row0_in = m0 + static_cast<int>(r0) < p.M;
            const bool row1_in = m0 + static_cast<int>(r1) < p.M;
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                int got = 1;
                if (lane == 0)
                    got = mbar_wait(bar_full + 8 * stage, phase, p.timeout_ns, abort_flag) ? 1 : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    if (lane == 0) fail(kRoleMeta);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();  // the MMAs that read this stage's columns completed
                const uint32_t e = sE + stage * Cfg::kEBytes;
                const uint4 w0 = ld_shared_v4_u32(e + 16u * r0);
                const uint4 w1 = ld_shared_v4_u32(e + 16u * r1);
                const uint32_t a[4] = {w0.x, w0.y, w0.z, w0.w};
                const uint32_t b[4] = {w1.x, w1.y, w1.z, w1.w};
                uint32_t t[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const bool word_in = kb * 4 + w < sp.words;
                    const uint32_t lo = (row0_in && word_in) ? (a[w] >> (16 * h)) & 0xFFFFu : kNeutral;
                    const uint32_t hi = (row1_in && word_in) ? (b[w] >> (16 * h)) & 0xFFFFu : kNeutral;
                    t[w] = lo | (hi << 16);
                }
                const uint32_t col = tmem_base + lane_addr + Cfg::kMetaCol0 +
                                     static_cast<uint32_t>(stage) * Cfg::kMetaStageCols;
#pragma unroll
                for (int w = 0; w < 4; ++w) tmem_st_x1(col + w * Cfg::kMetaSliceCols, t[w]);
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_meta + 8 * stage);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

}  // namespace tg
