// 2:4 structured-sparse GEMM on CTA pairs (tcgen05.mma.sp cta_group::2) for
// sm_103a:  C = epi(A · B) with A sparse, 256×256 output tiles per cluster.
//
// Same operation and operand formats as the one-CTA kernel (gemm_sparse.cuh:
// Ac = the kept values, E = 32-bit metadata words), the operation of "TileLang：
// 让GPU编程像Python一样简单的高性能计算新范式", section on sparse computation.
// What changes is the tile: each CTA of the pair (rank r) holds, per 128-k
// stage,
//   Ac rows [m0 + 128 r, +128) × 64 kept values   (one 16 KB box)
//   B cols  [n0 + 128 r, +128) × 128 k             (two 16 KB boxes)
//   E rows  [m0 + 128 r, +128) × 4 words           (one 2 KB box)
// and the even CTA issues 256×256×32 sparse MMAs over the pair.  Per SM this
// halves the operand bytes per MMA cycle of the 128×128 one-CTA tile, whose
// speed the L2 → SM bandwidth sets.
//
// Tensor memory (512 columns per CTA): one 256-column fp32 accumulator and,
// from column 256, one metadata slot of 64 columns per operand stage — each
// MMA's metadata column on a 16-column boundary.  Each CTA's tensor memory holds
// the metadata of its own 128 rows at the same column, in the lane layout of
// the one-CTA kernel.  With one accumulator the epilogue's tensor-memory
// reads of a tile are not overlapped with the next tile's MMAs (its global
// stores are).
//
// The metadata path is kept off the operand ring's critical path:
//   * E boxes are loaded (plain TMA, local barrier) three stages ahead of
//     the operands into their own 4-slot ring;
//   * tensor memory holds one metadata slot per operand stage: each CTA's
//     metadata warps write stage u's words into slot u % STAGES once the
//     MMAs of stage u - STAGES have completed (the stage's empty barrier),
//     then arrive on the even CTA's full barrier of the stage (the odd CTA's
//     warps with a relaxed remote arrive: tcgen05.wait::st has completed
//     their writes);
//   * so full[s] stands for the stage's operands and both CTAs' metadata,
//     while the operand loads wait only for their ring slot and run the
//     whole ring ahead of the MMAs.
// A single thread issuing every TMA copy of a stage would take longer than
// the stage's MMAs, so two threads (warps 0 and 10) share them: warp 0 the
// Ac box and the E box kEAhead stages ahead, warp 10 the two B boxes.
//
// Synchronisation (all waits bounded):
//   full[s]    even CTA: Ac and B bytes of both CTAs (pair TMA loads), the
//              producer's arrive and the 8 metadata warps of the pair;
//   empty[s]   each CTA: multicast commit after the MMAs of stage s (frees
//              the operand slot and the metadata slot);
//   efull[e]   each CTA: its own E box;
//   efree[e]   each CTA: its 4 metadata warps read E slot e;
//   tfull      each CTA: multicast commit at the end of a tile;
//   tempty     even CTA: the 8 epilogue warps of the pair read the tile.
// A cluster barrier after set-up and before exit brackets the work.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "gemm_persistent.cuh"
#include "gemm_sparse.cuh"
#include "sm103_ptx.cuh"
#include "tile_schedule.h"

namespace tg {

template <int STAGES_>
struct SparsePairCfg {
    static constexpr int STAGES = STAGES_;
    static constexpr int BM = 256;      // rows of C per cluster tile (128 per CTA)
    static constexpr int BN = 256;      // columns of C per cluster tile (B: 128 per CTA)
    static constexpr int BK = 128;      // dense-equivalent k per stage
    static constexpr int kThreads = 352;
    static constexpr int kESlots = 4;   // E ring
    static constexpr int kEAhead = 3;   // E boxes issued this many stages ahead
    static constexpr uint32_t kABytes = 128 * (BK / 2) * 2;  // 16 KB of kept values
    static constexpr uint32_t kBBytes = BK * 128 * 2;        // 32 KB: two 64-column boxes
    static constexpr uint32_t kEBytes = 128 * (BK / 32) * 4; // 2 KB of metadata
    static constexpr uint32_t kCBuf = 32 * 64 * 2;
    // staging buffers per epilogue warp: two, or one where a fourth operand
    // stage takes the room (plain epilogue only)
    static constexpr int kCBufs = STAGES >= 4 ? 1 : 2;
    static constexpr uint32_t kCBytes = 4 * kCBufs * kCBuf;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kMetaCol0 = BN;
    static constexpr uint32_t kMetaSlotCols = 64;
    static constexpr uint32_t kMetaSliceCols = 16;
    static constexpr uint32_t kBarBytes = 256;
    static constexpr uint32_t kSmemBytes = 1024 + STAGES * (kABytes + kBBytes) +
                                           kESlots * kEBytes + kCBytes + kBarBytes;
    static_assert(kMetaCol0 + kMetaSlotCols * STAGES <= kTmemCols,
                  "metadata columns exceed tensor memory");
    // E slot (u + kEAhead) % kESlots was last read for stage u + kEAhead -
    // kESlots <= u - 1, a read that follows the MMAs of stage u - 1 - STAGES;
    // those completed before stage u's operand slot was free, so the
    // producer's wait for the read (efree) is short.
    static_assert(kEAhead < kESlots, "E ring too shallow for the look-ahead");
    static_assert(8 * (2 * STAGES + 2 * kESlots) + 32 <= kBarBytes,
                  "barrier area too small");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeded");
};

// mbar_wait for a barrier that threads of the peer CTA arrive on (release at
// cluster scope): the successful wait acquires at cluster scope.
__device__ __forceinline__ uint32_t mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns,
                                                  const volatile int* abort_flag) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// Arrive on an mbarrier of the peer CTA without release semantics (no memory
// barrier): used where the signal only says "this thread's tensor-memory
// reads (or writes) are done" — tcgen05.wait::ld (wait::st) completed them
// before the arrive issues, and there is no generic-proxy memory whose
// visibility it would have to order.  A release arrive at cluster scope costs
// a memory barrier of about 1500 cycles.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// Early-release epilogue step: 64 accumulator columns of this thread's row
// (tensor memory at taddr, one load) → bias, activation → 32 packed 16-bit
// pairs (h[t]: columns 2t, 2t + 1).
template <typename T>
__device__ __forceinline__ void epilogue_pack64(uint32_t taddr, const EpilogueArgs& e, int relu,
                                                int col0, int N, uint32_t (&h)[32]) {
    uint32_t v[64];
    tmem_ld_x64(taddr, v);
    float x[64];
#pragma unroll
    for (int t = 0; t < 64; ++t) x[t] = __uint_as_float(v[t]);
    if (e.bias != nullptr) {
        if (e.bias_vec && col0 + 64 <= N) {
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
#pragma unroll
    for (int t = 0; t < 32; ++t) h[t] = Elem16<T>::pack2(x[2 * t], x[2 * t + 1]);
}

// Stage and store one 64-column chunk of packed 16-bit pairs through this
// warp's single 4 KB staging buffer, once the previous store has read it.
__device__ __forceinline__ void epilogue_store_one_buffer(const uint32_t (&h)[32], uint32_t cbuf,
                                                          const void* tmC, uint64_t policy,
                                                          int row0, int col0, int M, int N,
                                                          int lane) {
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
    const uint32_t row_addr = cbuf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        st_shared_v4(row_addr + ((static_cast<uint32_t>(c) ^ (lane & 7u)) << 4), h[4 * c],
                     h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (row0 < M && col0 < N) tma_store_2d_hint(tmC, cbuf, col0, row0, policy);
        bulk_commit_group();
    }
}

__device__ __forceinline__ void mma_f16_sp_pair(uint32_t d_tmem, uint64_t a_desc,
                                                uint64_t b_desc, uint32_t meta_tmem,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.sp.cta_group::2.kind::f16 [%0], %1, %2, [%3], %4, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(meta_tmem), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One stage (128 dense-equivalent k) of the pair: four sparse MMAs of 256 ×
// 256 × 32 and the release commit of the stage (its operand and metadata
// slots, multicast to both CTAs), issued by one elected lane of a converged
// warp in one block.  MMA k reads A 32 B further (ad + 2 k), B 4 KB further (bd +
// 256 k) and metadata 16 columns further.  first != 0: the first MMA
// overwrites D.  The issuing warp shares its scheduler with the metadata and
// epilogue warps; the single block keeps its instruction count per stage low.
__device__ __forceinline__ void sp_pair_stage_mma_elect(uint32_t d_tmem, uint64_t ad, uint64_t bd,
                                                        uint32_t meta, uint32_t idesc,
                                                        uint32_t first, uint32_t bar_stage) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 m;\n\t.reg .b64 a, b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.eq.b32 p, %5, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "@e tcgen05.mma.sp.cta_group::2.kind::f16 [%0], %1, %2, [%3], %4, p;\n\t"
        "add.u64 a, %1, 2;\n\tadd.u64 b, %2, 256;\n\tadd.u32 m, %3, 16;\n\t"
        "@e tcgen05.mma.sp.cta_group::2.kind::f16 [%0], a, b, [m], %4, t;\n\t"
        "add.u64 a, %1, 4;\n\tadd.u64 b, %2, 512;\n\tadd.u32 m, %3, 32;\n\t"
        "@e tcgen05.mma.sp.cta_group::2.kind::f16 [%0], a, b, [m], %4, t;\n\t"
        "add.u64 a, %1, 6;\n\tadd.u64 b, %2, 768;\n\tadd.u32 m, %3, 48;\n\t"
        "@e tcgen05.mma.sp.cta_group::2.kind::f16 [%0], a, b, [m], %4, t;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%6], %7;\n\t"
        "}" ::"r"(d_tmem),
        "l"(ad), "l"(bd), "r"(meta), "r"(idesc), "r"(first), "r"(bar_stage),
        "h"(static_cast<uint16_t>(0x3))
        : "memory");
}

// Walks this cluster's (tile, k block) sequence: stage u is k block u % kb of
// the cluster's tile u / kb (tiles cluster_id, cluster_id + nclusters, ...).
// The tile's block coordinates (three integer divisions) are computed once
// per tile, not per stage: the producer issues a stage every few hundred
// cycles.
struct StageIter {
    int tile, kb, m_blk, n_blk;
    const PersistentParams& p;
    int step;
    __device__ StageIter(int first_tile, const PersistentParams& p_, int step_)
        : tile(first_tile), kb(0), m_blk(0), n_blk(0), p(p_), step(step_) {
        coords();
    }
    __device__ void coords() {
        if (tile < p.num_tiles) {
            const TileCoord c = tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m);
            m_blk = c.m_blk;
            n_blk = c.n_blk;
        }
    }
    __device__ void next() {
        if (++kb == p.k_blocks) {
            kb = 0;
            tile += step;
            coords();
        }
    }
};

// EX = false: the plain epilogue only (no bias, no residual, 16-bit C); the
// other epilogue paths are compiled out.
template <int STAGES, typename T, bool EX = true>
__global__ void __launch_bounds__(352, 1)
    tg_gemm_sp24_pair(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmE,
                      const __grid_constant__ CUtensorMap tmC, const SparseParams sp) {
    using Cfg = SparsePairCfg<STAGES>;
    static_assert(Cfg::kCBufs == 2 || !EX, "one staging buffer per warp: plain epilogue only");
    constexpr int S = STAGES;
    constexpr int SE = Cfg::kESlots;
    const PersistentParams& p = sp.base;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base;
    const uint32_t sB = sA + S * Cfg::kABytes;
    const uint32_t sE = sB + S * Cfg::kBBytes;
    const uint32_t sC = sE + SE * Cfg::kEBytes;
    const uint32_t sBar = sC + Cfg::kCBytes;
    const uint32_t bar_full = sBar;                  // [S]
    const uint32_t bar_empty = bar_full + 8 * S;     // [S]
    const uint32_t bar_efull = bar_empty + 8 * S;    // [SE]
    const uint32_t bar_efree = bar_efull + 8 * SE;   // [SE]
    const uint32_t bar_tfull = bar_efree + 8 * SE;
    const uint32_t bar_tempty = bar_tfull + 8;
    const uint32_t bar_drain = bar_tempty + 8;
    const uint32_t slot_tmem = bar_drain + 8;
    uint32_t* const tmem_slot_ptr = reinterpret_cast<uint32_t*>(base_ptr + (slot_tmem - base));
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot_ptr + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster_id = static_cast<int>(blockIdx.x >> 1);
    const int nclusters = static_cast<int>(gridDim.x >> 1);
    // stages this cluster runs: its tiles × k blocks
    const int my_tiles =
        cluster_id < p.num_tiles ? (p.num_tiles - cluster_id + nclusters - 1) / nclusters : 0;
    const int U = my_tiles * p.k_blocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1 + 8);  // producer + metadata warps (even CTA's)
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int e = 0; e < SE; ++e) {
            mbar_init(bar_efull + 8 * e, 1);
            mbar_init(bar_efree + 8 * e, 4);
        }
        mbar_init(bar_tfull, 1);
        mbar_init(bar_tempty, 8);
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
        tmem_alloc_pair(slot_tmem, Cfg::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist and its tensor memory is allocated
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot_ptr;
    grid_dependency_wait();  // the previous kernel's writes are visible from here on
    grid_launch_dependents();

    auto fail = [&](unsigned int role) {
        atomicOr(&g_wait_timeout_flags, role);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer of Ac and E (both CTAs)
        if (lane == 0) {
            const uint64_t a_policy = policy_evict_last();
            uint32_t issued_mask = 0, issued_parity = 0;      // full[] phases armed here
            uint32_t e_issued_mask = 0, e_issued_parity = 0;  // efull[] phases armed here
            StageIter e_it(cluster_id, p, nclusters);
            int e_next = 0;  // next stage whose E box is issued
            // E box of stage e_next into slot e_next % SE, once the metadata
            // warps have read the slot's previous box (stage e_next - SE).
            auto issue_e = [&]() -> bool {
                const int ma = e_it.m_blk * Cfg::BM + static_cast<int>(rank) * 128;
                const int slot = e_next % SE;
                const uint32_t par = static_cast<uint32_t>(e_next / SE) & 1u;
                if (!mbar_wait(bar_efree + 8 * slot, par ^ 1u, p.timeout_ns, abort_flag))
                    return false;
                const uint32_t eb = bar_efull + 8 * slot;
                mbar_arrive_expect_tx(eb, Cfg::kEBytes);
                tma_load_2d(sE + slot * Cfg::kEBytes, &tmE, eb, e_it.kb * (Cfg::BK / 32), ma);
                e_issued_mask |= 1u << slot;
                e_issued_parity = (e_issued_parity & ~(1u << slot)) | (par << slot);
                e_it.next();
                ++e_next;
                return true;
            };
            // the first kEAhead slots are free: these waits return at once
            while (e_next < U && e_next < Cfg::kEAhead) issue_e();
            bool ok = true;
            StageIter it(cluster_id, p, nclusters);
            int stage = 0;
            uint32_t phase = 0;
            for (int u = 0; u < U; ++u, it.next()) {
                if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.timeout_ns, abort_flag)) {
                    fail(kRoleProducer);
                    ok = false;
                    break;
                }
                const int ma = it.m_blk * Cfg::BM + static_cast<int>(rank) * 128;
                if (leader)
                    mbar_arrive_expect_tx(bar_full + 8 * stage, 2 * (Cfg::kABytes + Cfg::kBBytes));
                const uint32_t fb = mapa_shared(bar_full + 8 * stage, 0);
                // kept values of A: reread by every column block of the raster
                // group, so kept in L2 ahead of B and C
                tma_load_2d_pair_hint(sA + stage * Cfg::kABytes, &tmA, fb, it.kb * (Cfg::BK / 2),
                                      ma, a_policy);
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (e_next < U && !issue_e()) {
                    fail(kRoleProducer);
                    ok = false;
                    break;
                }
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) {
                // Normal exit: every phase armed here was consumed (by the MMA
                // thread, and by this CTA's metadata warps), so these return at once.
                for (int s = 0; s < S; ++s)
                    if (leader && (issued_mask & (1u << s)))
                        if (!mbar_wait(bar_full + 8 * s, (issued_parity >> s) & 1u, p.timeout_ns,
                                       nullptr))
                            atomicOr(&g_wait_timeout_flags, kRoleDrain);
                for (int e = 0; e < SE; ++e)
                    if (e_issued_mask & (1u << e))
                        if (!mbar_wait(bar_efull + 8 * e, (e_issued_parity >> e) & 1u,
                                       p.timeout_ns, nullptr))
                            atomicOr(&g_wait_timeout_flags, kRoleDrain);
            } else if ((issued_mask | e_issued_mask) != 0) {
                // Abort: this CTA's last loads may be counted on a phase the
                // pair never finishes; give them a fixed, bounded grace period
                // (far above a TMA round trip) to land.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 1000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        if (leader) {
            // The whole warp runs the loop (warp-uniform control flow and
            // operands); one elected lane issues the MMAs and commits.  A
            // wait counts as met only if every lane saw it met.
            // sparse (bit 2), selector 0; A K-major, B MN-major; 256 × 256 over the pair
            constexpr uint32_t idesc =
                idesc_f16_f32(Cfg::BM, Cfg::BN, /*a_mn=*/false, /*b_mn=*/true,
                              Elem16<T>::kFmt) |
                (1u << 2);
            static_assert(Cfg::BK / 32 == 4 && Cfg::kMetaSliceCols == 16,
                          "sp_pair_stage_mma_elect issues four MMAs 16 metadata columns apart");
            // Descriptors of stage 0; a stage or k step only moves the start
            // address, the descriptor's low 14 bits (address / 16, and every
            // address here is below 256 KB), so it is a plain add.
            const uint64_t adesc0 = smem_desc_sw128(sA, 16, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(sB, 16384, 1024);
            constexpr uint64_t kAStep = Cfg::kABytes >> 4, kBStep = Cfg::kBBytes >> 4;
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int tile = cluster_id; ok && tile < p.num_tiles; tile += nclusters, ++it) {
                const bool te = mbar_wait_cluster(bar_tempty, (static_cast<uint32_t>(it) & 1u) ^ 1u,
                                                  p.timeout_ns, abort_flag);
                if (!__all_sync(0xffffffffu, te ? 1 : 0)) {
                    if (lane == 0) fail(kRoleMma);
                    break;
                }
                tc_fence_after_sync();
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    // the stage's operands, and both CTAs' metadata for it
                    const bool got =
                        mbar_wait(bar_full + 8 * stage, phase, p.timeout_ns, abort_flag);
                    if (!__all_sync(0xffffffffu, got ? 1 : 0)) {
                        if (lane == 0) fail(kRoleMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    sp_pair_stage_mma_elect(
                        tmem_base, adesc0 + static_cast<uint64_t>(stage) * kAStep,
                        bdesc0 + static_cast<uint64_t>(stage) * kBStep,
                        tmem_base + Cfg::kMetaCol0 +
                            static_cast<uint32_t>(stage) * Cfg::kMetaSlotCols,
                        idesc, kb == 0 ? 1u : 0u, bar_empty + 8 * stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (!(p.inject == 1 && it == 0)) {
                    __syncwarp();
                    if (lane == 0) mma_commit_pair_mc(bar_tfull, 0x3);
                }
            }
            __syncwarp();
            if (lane == 0) mma_commit_pair_mc(bar_drain, 0x1);
            const bool dr = mbar_wait(bar_drain, 0, p.timeout_ns, nullptr);
            if (!__all_sync(0xffffffffu, dr ? 1 : 0) && lane == 0)
                atomicOr(&g_wait_timeout_flags, kRoleDrain);
        }
    } else if (warp == 10) {
        // ------------------------------------------------------------ producer of B (both CTAs)
        if (lane == 0) {
            StageIter it(cluster_id, p, nclusters);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            bool issued = false;
            for (int u = 0; u < U; ++u, it.next()) {
                if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.timeout_ns, abort_flag)) {
                    fail(kRoleProducer);
                    ok = false;
                    break;
                }
                // Counted on the even CTA's full barrier like the Ac box; the
                // phase completes only when warp 0 of the even CTA has armed it.
                const int nb = it.n_blk * Cfg::BN + static_cast<int>(rank) * 128;
                const uint32_t fb = mapa_shared(bar_full + 8 * stage, 0);
                tma_load_2d_pair(sB + stage * Cfg::kBBytes, &tmB, fb, nb, it.kb * Cfg::BK);
                tma_load_2d_pair(sB + stage * Cfg::kBBytes + Cfg::kBBytes / 2, &tmB, fb, nb + 64,
                                 it.kb * Cfg::BK);
                issued = true;
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok && issued) {
                // Abort: bounded grace period for the last loads to land.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 1000000ull) {
                }
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const uint32_t cbuf = sC + static_cast<uint32_t>((warp - 2) * Cfg::kCBufs) * Cfg::kCBuf;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        const uint64_t c_policy = policy_evict_first();
        const uint32_t tempty_leader = mapa_shared(bar_tempty, 0);
        const bool early_release = !EX || (p.out_f32 == 0 && p.e.resid == nullptr);
        const EpilogueArgs epi_e = EX ? p.e : EpilogueArgs{};
        int buf = 0;
        int it = 0;
        for (int tile = cluster_id; tile < p.num_tiles; tile += nclusters, ++it) {
            const TileCoord tc = tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m);
            const int row0 = tc.m_blk * Cfg::BM + static_cast<int>(rank) * 128 + 32 * q;
            const int n0 = tc.n_blk * Cfg::BN;
            int ok = 1;
            if (lane == 0)
                ok = mbar_wait(bar_tfull, static_cast<uint32_t>(it) & 1u, p.timeout_ns,
                               abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) fail(kRoleEpilogue);
                break;
            }
            tc_fence_after_sync();
            if constexpr (Cfg::kCBufs == 1) {
                // One staging buffer: columns 0..63 go straight into it,
                // 64..255 into registers, then the accumulator is released
                // and the chunks are stored one after another.
                if (lane == 0) bulk_wait_group_read<0>();  // the buffer is free
                __syncwarp();
                const uint32_t row_off = static_cast<uint32_t>(lane) * 128u;
                {
                    uint32_t hp[32];
                    epilogue_pack64<T>(tmem_base + lane_addr, epi_e, p.relu, n0, p.N, hp);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(cbuf + row_off +
                                         ((static_cast<uint32_t>(u) ^ (lane & 7u)) << 4),
                                     hp[4 * u], hp[4 * u + 1], hp[4 * u + 2], hp[4 * u + 3]);
                }
                uint32_t h1[32], h2[32], h3[32];
                epilogue_pack64<T>(tmem_base + lane_addr + 64u, epi_e, p.relu, n0 + 64, p.N, h1);
                epilogue_pack64<T>(tmem_base + lane_addr + 128u, epi_e, p.relu, n0 + 128, p.N, h2);
                epilogue_pack64<T>(tmem_base + lane_addr + 192u, epi_e, p.relu, n0 + 192, p.N, h3);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (row0 < p.M && n0 < p.N) tma_store_2d_hint(&tmC, cbuf, n0, row0, c_policy);
                    bulk_commit_group();
                }
                epilogue_store_one_buffer(h1, cbuf, &tmC, c_policy, row0, n0 + 64, p.M, p.N, lane);
                epilogue_store_one_buffer(h2, cbuf, &tmC, c_policy, row0, n0 + 128, p.M, p.N, lane);
                epilogue_store_one_buffer(h3, cbuf, &tmC, c_policy, row0, n0 + 192, p.M, p.N, lane);
            } else if (early_release) {
                // 16-bit C without a residual: the row's 256 columns are read,
                // finished and rounded before anything is stored — columns
                // 0..127 straight into the two staging buffers (swizzled as
                // epilogue_store_packed lays them out), 128..255 into
                // registers — so the accumulator is released first.
                if (lane == 0) bulk_wait_group_read<0>();  // both buffers free
                __syncwarp();
                const uint32_t row_off = static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    uint32_t hp[32];
                    epilogue_pack64<T>(tmem_base + lane_addr + static_cast<uint32_t>(64 * j), epi_e,
                                       p.relu, n0 + 64 * j, p.N, hp);
                    const uint32_t rb = cbuf + static_cast<uint32_t>(j) * 4096u + row_off;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(rb + ((static_cast<uint32_t>(u) ^ (lane & 7u)) << 4),
                                     hp[4 * u], hp[4 * u + 1], hp[4 * u + 2], hp[4 * u + 3]);
                }
                uint32_t h2[32], h3[32];
                epilogue_pack64<T>(tmem_base + lane_addr + 128u, epi_e, p.relu, n0 + 128, p.N, h2);
                epilogue_pack64<T>(tmem_base + lane_addr + 192u, epi_e, p.relu, n0 + 192, p.N, h3);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (row0 < p.M && n0 + 64 * j < p.N)
                            tma_store_2d_hint(&tmC, cbuf + static_cast<uint32_t>(j) * 4096u,
                                              n0 + 64 * j, row0, c_policy);
                        bulk_commit_group();
                    }
                }
                buf = 0;
                epilogue_store_packed(h2, cbuf, buf, &tmC, c_policy, row0, n0 + 128, p.M, p.N,
                                      lane);
                epilogue_store_packed(h3, cbuf, buf, &tmC, c_policy, row0, n0 + 192, p.M, p.N,
                                      lane);
            } else {
#pragma unroll 1
                for (int j = 0; j < Cfg::BN / 64; ++j) {
                    uint32_t v0[32], v1[32];
                    const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(j * 64);
                    tmem_ld_x32(taddr, v0);
                    tmem_ld_x32(taddr + 32, v1);
                    if (j == Cfg::BN / 64 - 1) {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
                    }
                    float x[64];
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        x[t] = __uint_as_float(v0[t]);
                        x[32 + t] = __uint_as_float(v1[t]);
                    }
                    epilogue_math<T>(x, epi_e, p.relu, row0 + lane, n0 + 64 * j, p.M, p.N);
                    epilogue_store<T>(x, cbuf, buf, &tmC, c_policy, row0, n0 + 64 * j, p.M,
                                      p.N, lane, EX && p.out_f32 != 0);
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    } else {
        // ------------------------------------------------------------ metadata (warps 6..9, both CTAs)
        static_assert(Cfg::kThreads == 11 * 32, "warp roles: 0, 1, 2-5, 6-9, 10");
        // Lane L of this CTA's tensor memory (quarter warp % 4) takes rows
        // r0 = (L & ~15) | (L & 7) and r1 = r0 + 8 of the CTA's 128, k half
        // h = (L >> 3) & 1 of each of the stage's four 32-k words.
        const uint32_t L = 32u * static_cast<uint32_t>(warp & 3) + static_cast<uint32_t>(lane);
        const uint32_t r0 = (L & ~15u) | (L & 7u);
        const uint32_t r1 = r0 + 8u;
        const uint32_t h = (L >> 3) & 1u;
        const uint32_t lane_addr = (32u * static_cast<uint32_t>(warp & 3)) << 16;
        constexpr uint32_t kNeutral = 0x4444u;  // positions (0, 1) in every group of a half
        // The MMA thread reads these writes once the even CTA's full barrier
        // of the stage has the pair's 8 arrivals (and the operand bytes).  A
        // relaxed arrive suffices for the odd CTA: tcgen05.wait::st has
        // completed the writes before it issues, and no other memory is
        // handed over.
        const uint32_t full_leader = mapa_shared(bar_full, 0);
        StageIter it(cluster_id, p, nclusters);
        int eslot = 0, mslot = 0;
        uint32_t ephase = 0, mphase = 0;  // mslot: the stage's operand and metadata slot
        for (int u = 0; u < U; ++u, it.next()) {
            int got = 1;
            if (lane == 0)
                got = (mbar_wait(bar_efull + 8 * eslot, ephase, p.timeout_ns, abort_flag) &&
                       mbar_wait(bar_empty + 8 * mslot, mphase ^ 1u, p.timeout_ns, abort_flag))
                          ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                if (lane == 0) fail(kRoleMeta);
                break;
            }
            tc_fence_after_sync();  // the MMAs that read this slot completed
            const int m0 = it.m_blk * Cfg::BM + static_cast<int>(rank) * 128;
            const bool row0_in = m0 + static_cast<int>(r0) < p.M;
            const bool row1_in = m0 + static_cast<int>(r1) < p.M;
            const uint32_t e = sE + static_cast<uint32_t>(eslot) * Cfg::kEBytes;
            const uint4 w0 = ld_shared_v4_u32(e + 16u * r0);
            const uint4 w1 = ld_shared_v4_u32(e + 16u * r1);
            const uint32_t a[4] = {w0.x, w0.y, w0.z, w0.w};
            const uint32_t b[4] = {w1.x, w1.y, w1.z, w1.w};
            uint32_t t[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const bool word_in = it.kb * 4 + w < sp.words;
                const uint32_t lo = (row0_in && word_in) ? (a[w] >> (16 * h)) & 0xFFFFu : kNeutral;
                const uint32_t hi = (row1_in && word_in) ? (b[w] >> (16 * h)) & 0xFFFFu : kNeutral;
                t[w] = lo | (hi << 16);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_efree + 8 * eslot);  // the E slot is read
            const uint32_t col = tmem_base + lane_addr + Cfg::kMetaCol0 +
                                 static_cast<uint32_t>(mslot) * Cfg::kMetaSlotCols;
#pragma unroll
            for (int w = 0; w < 4; ++w) tmem_st_x1(col + w * Cfg::kMetaSliceCols, t[w]);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(bar_full + 8 * mslot);
                else
                    mbar_arrive_cluster_relaxed(full_leader + 8u * static_cast<uint32_t>(mslot));
            }
            if (++eslot == SE) {
                eslot = 0;
                ephase ^= 1u;
            }
            if (++mslot == S) {
                mslot = 0;
                mphase ^= 1u;
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // the peer no longer reads this CTA's memory or signals its barriers
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
}

}  // namespace tg
