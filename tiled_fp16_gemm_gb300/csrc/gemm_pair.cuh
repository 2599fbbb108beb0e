// Persistent FP16 GEMM on CTA pairs (tcgen05 cta_group::2) for sm_103a:
//   C = epi(A · B), 256×256 output tiles per cluster of two CTAs.
//
// Each CTA of the pair (rank r = 0, 1) owns, per stage of BK k, in its own
// shared memory:
//   A rows  [m0 + 128 r, m0 + 128 r + 128)  × BK k  (K-major, BK/64 boxes of 16 KB)
//   B cols  [n0 + 128 r, n0 + 128 r + 128)  × BK k  (MN-major, two boxes of 64 columns)
// at identical offsets.  The even CTA's single MMA thread issues
// 256×256×16 tcgen05.mma over the pair; result rows 128 r .. 128 r + 127 land
// in CTA r's TMEM (two 256-column fp32 accumulators per CTA).  Per SM this
// halves the operand bytes loaded per MMA cycle compared with a one-CTA
// 128×256 tile.  One MMA covers 128 tensor cycles of the SM, and each issue
// costs the MMA thread a large part of that, so the per-stage work of that
// thread (barrier wait, fence, commit) is spread over BK/16 MMAs.
//
// Synchronisation (all waits bounded):
//   full[s]     in the even CTA only: its producer arms it with the bytes of
//               both CTAs; both CTAs' TMA loads count their bytes on it.
//   empty[s]    in each CTA: the MMA thread's commit is multicast to both.
//   tmem_full   in each CTA: multicast commit at the end of a tile.
//   tmem_empty  in the even CTA: all 8 epilogue warps of the pair arrive.
// A cluster barrier after set-up (barriers initialised, TMEM allocated) and
// before exit (no peer still reads or signals this CTA) brackets the work.
//
// Work items (tile_schedule.h, pair_item): each pair walks its share of the
// full waves of tiles; the tiles of a last, partial wave may be shared out
// to otherwise idle pairs, as column halves or as k-pieces.  A column half is
// a 256×128 product over all of k: each CTA loads one 64-column box of B per
// stage and the MMA takes N = 128.  A k-piece's epilogue (pair_tail_piece)
// writes an fp32 partial and counts itself in; the last piece of a tile sums
// them in k order and stores C.
//
// Structure: producer warp / MMA warp / four epilogue warps as in the
// one-CTA kernel (gemm_persistent.cuh), which follows the warp-specialised
// TMA + mbarrier ring of "TileLang：比 Triton 低一层的 tile 语言", section
// "它生成了什么", re-designed around TMEM and CTA pairs.
#pragma once

#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "gemm_persistent.cuh"
#include "sm103_ptx.cuh"
#include "tile_schedule.h"

namespace tg {

template <int STAGES, int BK_ = 64>
struct PairCfg {
    static constexpr int BM = 256;  // rows of C per cluster tile (128 per CTA)
    static constexpr int BN = 256;  // columns of C per cluster tile
    static constexpr int BK = BK_;
    static_assert(BK % 64 == 0, "A arrives in 64-k boxes");
    static constexpr int kThreads = 192;
    static constexpr uint32_t kABytes = 128 * BK * 2;  // this CTA's A half
    static constexpr uint32_t kBBytes = 128 * BK * 2;  // this CTA's B half
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kCBuf = 32 * 64 * 2;
    static constexpr uint32_t kCBytes = 4 * 2 * kCBuf;
    static constexpr uint32_t kBarBytes = 256;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kSmemBytes =
        1024 + STAGES * kStageBytes + kCBytes + kBarBytes;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeded");
    // a split tail tile's reduction borrows 48 KB of the ring per epilogue warp
    static_assert(STAGES * kStageBytes >= 4 * 48 * 1024, "ring too small for the reduction");
};

// Partial slots of split tail tiles: per cluster, 8 warp regions (rank × lane
// quarter) of 32 rows × 256 columns.  Inside a region, column group g (4
// columns) of row `lane` is the float4 at ((g · 32) + lane) · 4, so each warp
// store instruction covers 512 contiguous bytes and each 64-column chunk is
// 8 KB of contiguous floats.
constexpr int64_t kPairWarpFloats = 32 * 256;
constexpr int64_t kPairSlotFloats = 8 * kPairWarpFloats;  // 256 KB
constexpr uint32_t kPairChunkBytes = 64 * 32 * 4;         // one 64-column chunk of a region
constexpr uint32_t kPairRedBytes = 48 * 1024;             // per epilogue warp, in the ring

// Epilogue of one warp for a piece of a split tail tile (see tile_schedule.h).
// A piece is always its cluster's last item, so the operand ring is idle and
// the accumulator is not overwritten after its tmem_full.  The warp writes its
// partial to the cluster's slot and adds one to the counter of (tail tile,
// rank, quarter).  The warp that brings the counter to p.split sums the
// tile's pieces in k order (piece 0 first): its own from tensor memory, the
// others bulk-copied two chunks at a time into its 48 KB share of the ring
// (red: its own barrier there).  It then applies the epilogue, stores C and
// zeroes the counter.  Returns false if a bulk copy did not land in time.
template <typename T, bool EX>
__device__ __forceinline__ bool pair_tail_piece(const PersistentParams& p, uint32_t taddr,
                                                uint32_t tempty, int cluster_id, uint32_t rank,
                                                int q, int lane, uint32_t red_buf,
                                                uint32_t red_bar, uint32_t cbuf, int& buf,
                                                const void* tmC, uint64_t c_policy, int row0,
                                                int n0) {
    const int64_t region = static_cast<int64_t>(rank * 4 + static_cast<uint32_t>(q)) *
                           kPairWarpFloats;
    float* const mine = p.ws + static_cast<int64_t>(cluster_id) * kPairSlotFloats + region;
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
        uint32_t v[64];
        tmem_ld_x64(taddr + static_cast<uint32_t>(64 * j), v);
#pragma unroll
        for (int g = 0; g < 16; ++g)
            __stcg(reinterpret_cast<float4*>(mine + ((16 * j + g) * 32 + lane) * 4),
                   make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                               __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3])));
    }
    fence_proxy_async_global();  // the stores come before the reader's bulk copies of them
    __threadfence();
    __syncwarp();
    const int S = p.split;
    const int tail_tile = cluster_id / S;
    const int own = cluster_id - tail_tile * S;  // this piece's place in k order
    int last = 0;
    if (lane == 0) {
        uint32_t* cnt = p.counters + 8 * tail_tile + static_cast<int>(rank) * 4 + q;
        const uint32_t before = atomic_add_acq_rel_gpu(cnt, 1u);
        last = before + 1 == static_cast<uint32_t>(S) ? 1 : 0;
        if (last) *cnt = 0u;  // zero again for the next launch
    }
    bool ok = true;
    if (__shfl_sync(0xffffffffu, last, 0)) {
        __threadfence();
        // the other pieces' partials, observed through the acquire above, are
        // read below by bulk copies (the async proxy)
        if (lane == 0) fence_proxy_async_global();
        const float* const first =
            p.ws + static_cast<int64_t>(tail_tile) * S * kPairSlotFloats + region;
#pragma unroll 1
        for (int half = 0; half < 2 && ok; ++half) {
            // the other pieces' chunks 2·half and 2·half + 1
            if (lane == 0) {
                fence_proxy_async_smem();  // earlier reads of the buffer come first
                mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>(S - 1) * 2u *
                                                   kPairChunkBytes);
                int o = 0;
                for (int s = 0; s < S; ++s) {
                    if (s == own) continue;
                    for (int jj = 0; jj < 2; ++jj)
                        bulk_load(red_buf + static_cast<uint32_t>(2 * o + jj) * kPairChunkBytes,
                                  first + s * kPairSlotFloats + (2 * half + jj) * 2048,
                                  kPairChunkBytes, red_bar);
                    ++o;
                }
                // copies in flight must land before anything else: no abort
                ok = mbar_wait(red_bar, static_cast<uint32_t>(half), p.timeout_ns, nullptr);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            mbar_wait(red_bar, static_cast<uint32_t>(half), p.timeout_ns, nullptr);  // lanes 1..31
#pragma unroll 1
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * half + jj;
                uint32_t v[64];
                tmem_ld_x64(taddr + static_cast<uint32_t>(64 * j), v);
                float x[64];
                int o = 0;
                for (int s = 0; s < S; ++s) {
                    if (s == own) {
#pragma unroll
                        for (int t = 0; t < 64; ++t)
                            x[t] = s == 0 ? __uint_as_float(v[t]) : x[t] + __uint_as_float(v[t]);
                    } else {
                        const uint32_t src = red_buf +
                                             static_cast<uint32_t>(2 * o + jj) * kPairChunkBytes +
                                             static_cast<uint32_t>(lane) * 16u;
#pragma unroll
                        for (int g = 0; g < 16; ++g) {
                            const float4 a = ld_shared_f4(src + static_cast<uint32_t>(g) * 512u);
                            x[4 * g] = s == 0 ? a.x : x[4 * g] + a.x;
                            x[4 * g + 1] = s == 0 ? a.y : x[4 * g + 1] + a.y;
                            x[4 * g + 2] = s == 0 ? a.z : x[4 * g + 2] + a.z;
                            x[4 * g + 3] = s == 0 ? a.w : x[4 * g + 3] + a.w;
                        }
                        ++o;
                    }
                }
                epilogue_math<T>(x, EX ? p.e : EpilogueArgs{}, p.relu, row0 + lane, n0 + 64 * j,
                                 p.M, p.N);
                epilogue_store<T>(x, cbuf, buf, tmC, c_policy, row0, n0 + 64 * j, p.M, p.N,
                                  lane, EX && p.out_f32 != 0);
            }
            __syncwarp();  // every lane is done reading the buffer
        }
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(tempty);
    return ok;
}

// EX = false: the plain epilogue only (no bias, no residual, 16-bit C); the
// other epilogue paths are compiled out.
template <int STAGES, typename T = __half, int BK_ = 64, bool EX = true>
__global__ void __launch_bounds__(192, 1)
    tg_gemm_f16_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const PersistentParams p) {
    using Cfg = PairCfg<STAGES, BK_>;
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
    const uint32_t bar_full = sBar;
    const uint32_t bar_empty = sBar + 8 * STAGES;
    const uint32_t bar_tfull = sBar + 16 * STAGES;
    const uint32_t bar_tempty = bar_tfull + 16;
    const uint32_t bar_drain = bar_tempty + 16;
    const uint32_t bar_red = bar_drain + 8;  // [4] split tail tiles: the epilogue warps' copies
    const uint32_t slot_tmem = bar_red + 32;
    uint32_t* const tmem_slot_ptr = reinterpret_cast<uint32_t*>(base_ptr + (slot_tmem - base));
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot_ptr + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster_id = static_cast<int>(blockIdx.x >> 1);
    const int nclusters = static_cast<int>(gridDim.x >> 1);
    const int items = pair_item_count(cluster_id, p.num_tiles, nclusters, p.split, p.split_n);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + 8 * a, 1);
            mbar_init(bar_tempty + 8 * a, 8);
        }
        mbar_init(bar_drain, 1);
        for (int e = 0; e < 4; ++e) mbar_init(bar_red + 8 * e, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(slot_tmem, Cfg::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist and its TMEM is allocated
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot_ptr;
    // No L2 prefetch of the first operand tiles here (the one-CTA and skinny
    // kernels issue one before the dependency wait): timed back to back, it
    // took 2048^3 from 15.6 to 16.1 us and left 4096^3 and 8192×28672×4096
    // unchanged.
    grid_dependency_wait();  // the previous kernel's writes are visible from here on
    grid_launch_dependents();

    auto fail = [&](unsigned int role) {
        atomicOr(&g_wait_timeout_flags, role);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            // A panels are reread by every column block of their raster group
            // (about 24 waves of tiles on the 8192-row MLP shape): keep them
            // in L2 ahead of B tiles (reread within a wave) and C (evict-first).
            const uint64_t a_policy = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            uint64_t last_issue = 0;
            for (int i = 0; ok && i < items; ++i) {
                int tile, kb0, kb1, half;
                pair_item(cluster_id, i, p.num_tiles, nclusters, p.split, p.split_n, p.k_blocks,
                          &tile, &kb0, &kb1, &half);
                const TileCoord tc = tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m);
                const int ma = tc.m_blk * 256 + static_cast<int>(rank) * 128;
                // this CTA's B columns: 128 of a whole tile, 64 of a column half
                const int nb = half < 0 ? tc.n_blk * 256 + static_cast<int>(rank) * 128
                                        : tc.n_blk * 256 + half * 128 + static_cast<int>(rank) * 64;
                const uint32_t stage_tx =
                    half < 0 ? 2 * Cfg::kStageBytes : 2 * (kABytes + kBBytes / 2);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.timeout_ns, abort_flag)) {
                        fail(kRoleProducer);
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, stage_tx);
                    const uint32_t fb = mapa_shared(bar_full + 8 * stage, 0);
#pragma unroll
                    for (int i = 0; i < BK / 64; ++i)
                        tma_load_2d_pair_hint(sA + stage * kABytes + 16384 * i, &tmA, fb,
                                              kb * BK + 64 * i, ma, a_policy);
                    tma_load_2d_pair(sB + stage * kBBytes, &tmB, fb, nb, kb * BK);
                    if (half < 0)
                        tma_load_2d_pair(sB + stage * kBBytes + kBBytes / 2, &tmB, fb, nb + 64,
                                         kb * BK);
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (ok && leader) {
                // Normal exit: every phase armed here completed (the MMA
                // thread consumed it), so these waits return at once.
                for (int s = 0; s < STAGES; ++s)
                    if (issued_mask & (1u << s))
                        if (!mbar_wait(bar_full + 8 * s, (issued_parity >> s) & 1u, p.timeout_ns,
                                       nullptr))
                            atomicOr(&g_wait_timeout_flags, kRoleDrain);
            } else if (!ok && issued_mask != 0) {
                // Abort: completion of this CTA's last loads may be counted on
                // a phase the pair never finishes, so give them a fixed,
                // bounded grace period (far above a TMA round trip) to land.
                last_issue = globaltimer_ns();
                while (globaltimer_ns() - last_issue < 1000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        if (leader) {
            // The whole warp runs the loop (warp-uniform control flow and
            // operands); one elected lane issues each stage's MMAs and
            // commit.  A wait counts as met only if every lane saw it met.
            static_assert(BK == 128, "pair_stage_mma_elect issues 128 k per stage");
            constexpr uint32_t idesc =
                idesc_f16_f32(256, 256, /*a_mn=*/false, /*b_mn=*/true, Elem16<T>::kFmt);
            // a column half: N = 128, 64 columns of B in each CTA
            constexpr uint32_t idesc_half =
                idesc_f16_f32(256, 128, /*a_mn=*/false, /*b_mn=*/true, Elem16<T>::kFmt);
            auto warp_wait = [&](uint32_t bar, uint32_t parity, const volatile int* ab) {
                const bool r = mbar_wait(bar, parity, p.timeout_ns, ab);
                return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
            };
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (; ok && it < items; ++it) {
                int tile, kb0, kb1, half;
                pair_item(cluster_id, it, p.num_tiles, nclusters, p.split, p.split_n, p.k_blocks,
                          &tile, &kb0, &kb1, &half);
                const uint32_t id = half < 0 ? idesc : idesc_half;
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!warp_wait(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag)) {
                    if (lane == 0) fail(kRoleMma);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!warp_wait(bar_full + 8 * stage, phase, abort_flag)) {
                        if (lane == 0) fail(kRoleMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    // A: 64-k boxes of 16 KB; B: the two column boxes kBBytes/2 apart
                    pair_stage_mma_elect(d_tmem, smem_desc_sw128(sA + stage * kABytes, 16, 1024),
                                         smem_desc_sw128(sB + stage * kBBytes, kBBytes / 2, 1024),
                                         id, kb == kb0 ? 1u : 0u, bar_empty + 8 * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (!(p.inject == 1 && it == 0)) {
                    __syncwarp();
                    if (lane == 0) mma_commit_pair_mc(bar_tfull + 8 * acc, 0x3);
                }
            }
            __syncwarp();
            if (lane == 0) mma_commit_pair_mc(bar_drain, 0x1);
            if (!warp_wait(bar_drain, 0, nullptr) && lane == 0)
                atomicOr(&g_wait_timeout_flags, kRoleDrain);
        }
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const uint32_t cbuf = sC + static_cast<uint32_t>((warp - 2) * 2) * Cfg::kCBuf;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        const uint64_t c_policy = policy_evict_first();  // C is written once, never reread
        int buf = 0;
        int it = 0;
        for (; it < items; ++it) {
            int tile, kb0, kb1, half;
            pair_item(cluster_id, it, p.num_tiles, nclusters, p.split, p.split_n, p.k_blocks,
                      &tile, &kb0, &kb1, &half);
            const TileCoord tc = tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m);
            const int row0 = tc.m_blk * 256 + static_cast<int>(rank) * 128 + 32 * q;
            const int n0 = tc.n_blk * 256 + (half < 0 ? 0 : 128 * half);
            const int chunks = half < 0 ? 4 : 2;  // of 64 columns
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
            if (kb1 - kb0 < p.k_blocks) {
                // A piece of a split tail tile: this warp's 32 rows × 256
                // columns of fp32 partial go to the cluster's slot; the warp
                // whose add completes the tile's count sums the slots.
                const uint32_t e = static_cast<uint32_t>(warp - 2);
                if (!pair_tail_piece<T, EX>(p, tmem_base + lane_addr + static_cast<uint32_t>(acc * 256),
                                        mapa_shared(bar_tempty + 8 * acc, 0), cluster_id, rank,
                                        q, lane, sA + e * kPairRedBytes, bar_red + 8 * e, cbuf,
                                        buf, &tmC, c_policy, row0, n0) &&
                    lane == 0)
                    fail(kRoleEpilogue);
                continue;
            }
#pragma unroll 1
            for (int j = 0; j < chunks; ++j) {
                uint32_t v0[32], v1[32];
                const uint32_t taddr =
                    tmem_base + lane_addr + static_cast<uint32_t>(acc * 256 + j * 64);
                tmem_ld_x32(taddr, v0);
                tmem_ld_x32(taddr + 32, v1);
                if (j == chunks - 1) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(bar_tempty + 8 * acc, 0));
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
    cluster_sync();  // the peer no longer reads this CTA's smem or signals its barriers
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
}

}  // namespace tg
