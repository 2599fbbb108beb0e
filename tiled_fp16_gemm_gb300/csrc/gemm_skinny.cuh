// Skinny FP16 GEMM (M ≤ 128) for sm_103a:  C = epi(A · B), bandwidth bound.
//
// With few rows of C the 128-row tensor-core tile would mostly multiply
// padding, and ceil(N/BN) tiles leave most SMs idle while B (the large
// operand) streams from HBM.  So this kernel computes the transposed product
//     C^T (N×M) = B^T (N×K) · A^T (K×M)
// with N as the 128-row MMA dimension and Mp = roundup(M, 16) as the MMA
// N dimension:
//   MMA A operand = B^T tile, 128 n × BK k, read MN-major from row-major B;
//   MMA B operand = A tile,   Mp m × BK k, K-major from row-major A;
//   D (TMEM)      = 128 lanes (n) × Mp columns (m), fp32.
// BK (k per unit) is a parameter of the ring shape; both shapes use 64.  On
// the 64×16384×8192 workload, units of 128 k (4 stages of 48 KB) and of 256
// k (2 stages of 96 KB: B in 32 KB boxes) measured 52.5 and 53.3 µs against
// 51.7 µs for 64 k (9 stages of 24 KB).
//
// Split-K over "units" (tile, k-block), numbered tile-major.  CTA c of G owns
// the contiguous unit range [U·c/G, U·(c+1)/G), so every SM streams the same
// number of B bytes.  A range is cut at tile edges into segments:
//   FULL     the whole k range of a tile: the epilogue writes C directly;
//   piece    a segment that starts or ends inside its tile.  The tile's
//            pieces lie in CTAs c_head .. c_tail in k order: the head's is its
//            last segment (k = 0 onwards), every other one is its CTA's first
//            segment.  Each epilogue warp writes its 32 columns of the fp32
//            partial to its CTA's slot for it (first segment: slot 2c; head:
//            slot 2c + 1), then adds one to counter[4 c_head + warp quarter].
//            The warp that brings the counter to the number of pieces adds the
//            slots in k order (head first), applies the epilogue, writes C and
//            zeroes the counter, so counters are zero between launches.
// The epilogue (bias, ReLU, residual, output type) is applied per element by
// the thread holding column n: C[m][n] = out(act(acc + bias[n]) + R[m][n]),
// with plain stores (consecutive threads write consecutive n).
// The summation order is fixed by the sizes alone, whichever piece finishes
// last, so results are deterministic.  No CTA waits for another, so the
// launch needs no co-residency guarantee (and no cooperative launch); the
// waits inside a CTA are bounded.
//
// The pages do not describe a split-K or swap-AB variant; this is the plain
// reading of "measure the bandwidth and compute ceilings first"
// ("TileLang：比 Triton 低一层的 tile 语言", section "工程上的几个注意点"):
// a 64×16384×8192 product is bound by streaming B, so the kernel is shaped to
// keep every SM's TMA unit busy on B.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "gemm_persistent.cuh"
#include "mxfp4.cuh"
#include "sm103_ptx.cuh"
#include "tile_schedule.h"
#include "tgemm.h"

namespace tg {

// B^T tile of one unit: two boxes of 64 columns × BK k.
__host__ __device__ constexpr uint32_t skinny_b_bytes(int bk) {
    return 128u * static_cast<uint32_t>(bk) * 2u;
}

// Two ring shapes, both about 220 KB of shared memory: A slots sized for
// Mp ≤ 64 (24 KB stages, 9 deep: 144 KB of B in flight per SM) or for
// Mp ≤ 128 (32 KB stages, 6 deep).  A stage of BK k holds B^T as two boxes
// of 64 columns × BK k and the A tile as BK/64 boxes of 64 k.
template <int STAGES, int MP_MAX, int BK_>
struct SkinnyCfg {
    static constexpr int kStages = STAGES;
    static constexpr int kBK = BK_;
    static constexpr uint32_t kASlot = MP_MAX * BK_ * 2;
    static constexpr uint32_t kStageBytes = skinny_b_bytes(BK_) + kASlot;
    static constexpr uint32_t kSmemBytes = 1024 + STAGES * kStageBytes + 256;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeded");
};
using SkinnyNarrow = SkinnyCfg<9, 64, 64>;
using SkinnyWide = SkinnyCfg<6, 128, 64>;
// MXFP4 B (M ≤ 128 weight streaming), units of kMxBK = 128 k.
//   Raw ring (four producer threads): per unit, two 128 n × 64 k tiles of
//     packed codes (128 rows × 32 bytes each, TMA 32-byte swizzle) and their
//     scales (4 rows × 128 bytes).  The codes are the HBM stream; 8 stages
//     (68 KB) keep enough of it in flight per SM.
//   A ring (one producer thread, its own depth): the unit's activation tile
//     (from L2, re-read by every CTA).  A stage is released by a commit of
//     its own once the unit's MMAs have completed.  Tied to the operand
//     stages, a 4-deep ring let each tile be requested only 4 units ahead,
//     and its L2 round trip under the HBM stream then set the pace.
//   Converters (kMxGroups groups of four warps, one per tensor-memory lane
//     quarter, taking units in turn): thread n owns weight column n of the
//     tile, loads its 128 k of codes and the unit's scales into registers
//     (which frees the raw stage), decodes them into fp16 and writes them
//     with tcgen05.st straight into the unit's operand stage (the weight
//     tile is the A operand of the swapped product), so decoded weights
//     never pass through shared memory.
//   Tensor memory: two accumulators of MP_MAX columns, then operand stages
//     of 64 columns in the rest (6 for Mp ≤ 64, 4 for Mp ≤ 128).
// The MMA thread waits for the unit's operand stage (decoded) and its A
// stage (landed), issues 8 MMAs and commits twice: the operand stage back to
// the converters, the A stage back to its producer.
constexpr int kMxBK = 128;                       // k per MXFP4 unit
constexpr uint32_t kMxCodeBox = 128 * 32;        // one 64-k tile of codes
constexpr uint32_t kMxRawBytes = (kMxBK / 64) * kMxCodeBox;
constexpr uint32_t kMxScaleBytes = (kMxBK / 32) * 128;
constexpr uint32_t kMxOpCols = kMxBK / 2;        // tensor-memory columns per operand stage
// Converter groups of four warps (one per tensor-memory lane quarter, both
// 64-k halves of a unit each) or eight (two per quarter, one half each).
constexpr int kMxGroups = 3;
constexpr int kMxGroupWarps = 4;
constexpr int kMxHalvesPerWarp = 8 / kMxGroupWarps;
constexpr int kMxConvWarps = kMxGroupWarps * kMxGroups;
// Two MMA warps take a segment's units in turn, each into its own
// accumulator; the epilogue adds the two (first warp's first).  One warp's
// wait, issue and loop per unit took about twice the tensor pipe's 256
// cycles of MMA work, and its MMA issue blocks until the pipe takes them, so
// with one warp the pipe idled for the rest.
constexpr int kMxMmaWarps = 2;
constexpr uint32_t kMxTmemCols = 512;
constexpr int kMxRawStages = 8;
__host__ __device__ constexpr int mx_raw_stages(int mp_max) { return (void)mp_max, kMxRawStages; }
// first tensor-memory column of the operand stages: after the accumulators
// (one per MMA warp; a CTA's unit range spans at most a few tile segments,
// so they are not double-buffered)
__host__ __device__ constexpr uint32_t mx_op_col0(int mp_max) { return kMxMmaWarps * mp_max; }
__host__ __device__ constexpr int mx_op_stages(int mp_max) {
    return static_cast<int>((kMxTmemCols - mx_op_col0(mp_max)) / kMxOpCols);
}
constexpr uint32_t kMxBarBytes = 1024;
template <int MP_MAX>
struct SkinnyMxCfg {
    static constexpr int kStages = mx_op_stages(MP_MAX);  // tensor-memory operand stages
    static constexpr int kRawStages = kMxRawStages;
    static constexpr uint32_t kASlot = MP_MAX * kMxBK * 2;
    static constexpr int kAStages = MP_MAX <= 64 ? 8 : 4;  // 128 KB of activation tiles
    static constexpr uint32_t kStageBytes = 0;  // no shared-memory operand ring
    static constexpr uint32_t kRawStageBytes = kMxRawBytes + kMxScaleBytes;
    static constexpr uint32_t kSmemBytes =
        1024 + kRawStages * kRawStageBytes + kAStages * kASlot + kMxBarBytes;
    static_assert(mx_op_col0(MP_MAX) + kMxOpCols * kStages <= kMxTmemCols,
                  "operand stages exceed tensor memory");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeded");
    // barriers: full/empty/dec per operand stage, rfull/rempty per raw stage,
    // afull/aempty per A stage, two tfull, two tempty, drain, TMEM slot + flag
    static_assert(8 * (3 * kStages + 2 * kRawStages + 2 * kAStages) + 48 <= kMxBarBytes,
                  "barrier area too small");
};
using SkinnyMxNarrow = SkinnyMxCfg<64>;
using SkinnyMxWide = SkinnyMxCfg<128>;
constexpr unsigned int kRoleConvert = 16u;

// Load issue is split over several producer threads (one per warp): one
// thread's loop of slot wait, transaction arming and TMA issue costs a few
// hundred cycles per unit whatever the box size, which alone would cap a
// skinny kernel far below HBM bandwidth.  Producer p takes the units of local
// index i ≡ p (mod count); the count divides the ring depth, so each ring
// stage always belongs to the same producer.
__host__ __device__ constexpr int skinny_producers(int ring) {
    return ring % 4 == 0 ? 4 : (ring % 3 == 0 ? 3 : (ring % 2 == 0 ? 2 : 1));
}
// Threads of a skinny kernel: producer 0, MMA, 4 epilogue warps, the
// converter warps and the second MMA warp (MXFP4), producers 1 .. count - 1,
// then (MXFP4) the producer of the A ring.
__host__ __device__ constexpr int skinny_threads(int stages, int mp_max, bool qb) {
    return 32 * (6 + (qb ? kMxConvWarps + 2 : 0) +
                 skinny_producers(qb ? mx_raw_stages(mp_max) : stages) - 1);
}
constexpr uint32_t kSkTmemCols = 256;        // two accumulators of up to 128 columns
constexpr int64_t kSkSlotFloats = 128 * 128;  // one partial: Mp ≤ 128 rows × 128 n
constexpr int kSkMinUnitsPerCta = 8;

struct SkinnyParams {
    int32_t M, N, K, Mp;
    int32_t tiles_n, k_blocks;
    int64_t total_units;
    int32_t relu, inject;
    uint64_t timeout_ns;
    void* C;  // T*: the kernel's element type
    int64_t ldc;
    float* ws;            // two partial slots per CTA
    uint32_t* counters;   // four piece counters per CTA (zero between launches)
    EpilogueArgs e;       // bias / residual (null: none)
    int32_t out_f32 = 0;  // 1: C is fp32
};

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}


// Columns [a, a + 16) and [b, b + 16) of this warp's lane quarter (two
// accumulators) in one round trip: both loads, then one wait.
__device__ __forceinline__ void tmem_ld2_x16(uint32_t a, uint32_t b, uint32_t (&r)[16],
                                             uint32_t (&s)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(s[0]), "=r"(s[1]), "=r"(s[2]), "=r"(s[3]),
          "=r"(s[4]), "=r"(s[5]), "=r"(s[6]), "=r"(s[7]), "=r"(s[8]), "=r"(s[9]), "=r"(s[10]),
          "=r"(s[11]), "=r"(s[12]), "=r"(s[13]), "=r"(s[14]), "=r"(s[15])
        : "r"(a), "r"(b)
        : "memory");
}

// The kernel body shared by the fp16/bf16 kernel (QB = false: B^T tiles by
// TMA) and the MXFP4 kernel (QB = true: B^T tiles decoded by warps 6..13).
// EX = false: the plain epilogue only (no bias, no residual, 16-bit C), with a
// short store loop; the other epilogue paths are compiled out.
template <int STAGES, int MP_MAX, typename T, bool QB, int BK = 64, bool EX = true>
__device__ __forceinline__ void skinny_body(const CUtensorMap* tmB, const CUtensorMap* tmA,
                                            const CUtensorMap* tmS, const SkinnyParams& p) {
    static_assert(BK % 64 == 0 && (!QB || BK == kMxBK), "MXFP4 units are kMxBK");
    constexpr int kSkStages = STAGES;
    constexpr uint32_t kSkBBytes = skinny_b_bytes(BK);
    constexpr uint32_t kABox = MP_MAX * 64 * 2;   // one 64-k box of the A tile (≤ MP_MAX rows)
    constexpr uint32_t kSkASlot = kABox * (BK / 64);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    constexpr int kRaw = QB ? mx_raw_stages(MP_MAX) : 0;  // raw ring depth (QB)
    constexpr int kAS = QB ? SkinnyMxCfg<MP_MAX>::kAStages : 0;  // A ring depth (QB)
    constexpr int kARing = QB ? kAS : kSkStages;          // A slots: own ring, or with B
    // tensor-memory columns: accumulator stride, first operand-stage column (QB)
    constexpr uint32_t kAccStride = QB ? static_cast<uint32_t>(MP_MAX) : 128u;
    constexpr uint32_t kOpCol0 = QB ? mx_op_col0(MP_MAX) : 0u;
    // MMA warps, and accumulator buffers per MMA warp (segments alternate
    // over the buffers): accumulator (buffer b, warp m) is number b·kMW + m
    constexpr int kMW = QB ? kMxMmaWarps : 1;
    constexpr int kBufs = QB ? 1 : 2;
    constexpr int kBRing = QB ? 0 : kSkStages;            // B^T tiles in shared memory
    const uint32_t sB = base;                             // [kBRing] B^T tiles
    const uint32_t sA = sB + kBRing * kSkBBytes;          // [kARing] A tiles
    // QB only: [raw stages] packed codes, [raw stages] scales
    const uint32_t sRaw = sA + kARing * kSkASlot;
    const uint32_t sScl = sRaw + kRaw * kMxRawBytes;
    const uint32_t sBar = sScl + kRaw * kMxScaleBytes;
    const uint32_t bar_full = sBar;                       // [stages] A and B landed (fp16 B)
    const uint32_t bar_empty = sBar + 8 * kSkStages;      // [stages] MMA done with the stage
    const uint32_t bar_dec = sBar + 16 * kSkStages;       // QB: [stages] B^T decoded
    const uint32_t bar_rfull = bar_dec + (QB ? 8 * kSkStages : 0);  // QB: [raw] landed
    const uint32_t bar_rempty = bar_rfull + 8 * kRaw;     // QB: [raw] decoded
    const uint32_t bar_afull = bar_rempty + 8 * kRaw;     // QB: [A stages] landed
    const uint32_t bar_aempty = bar_afull + 8 * kAS;      // QB: [A stages] MMAs done
    const uint32_t bar_tfull = bar_aempty + 8 * kAS;
    const uint32_t bar_tempty = bar_tfull + 16;
    const uint32_t bar_drain = bar_tempty + 16;
    const uint32_t slot_tmem = bar_drain + 8;
    uint32_t* const tmem_slot_ptr = reinterpret_cast<uint32_t*>(base_ptr + (slot_tmem - base));
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot_ptr + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t U = p.total_units;
    const int64_t KB = p.k_blocks;
    const int64_t u_begin = unit_begin(blockIdx.x, G, U);
    const int64_t u_end = unit_begin(blockIdx.x + 1, G, U);
    const uint32_t a_bytes = static_cast<uint32_t>(p.Mp) * 128u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSkStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
            if (QB) mbar_init(bar_dec + 8 * s, kMxGroupWarps);  // the warps of one group
        }
        if (QB) {
            for (int r = 0; r < kRaw; ++r) {
                mbar_init(bar_rfull + 8 * r, 1);
                mbar_init(bar_rempty + 8 * r, kMxGroupWarps);  // the group's warps
            }
            for (int a = 0; a < kAS; ++a) {
                mbar_init(bar_afull + 8 * a, 1);
                mbar_init(bar_aempty + 8 * a, 1);
            }
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + 8 * a, kMW);  // one commit per MMA warp
            mbar_init(bar_tempty + 8 * a, 4);
        }
        mbar_init(bar_drain, kMW);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(tmA);
        tma_prefetch_desc(tmB);
        if (QB) tma_prefetch_desc(tmS);
    }
    constexpr uint32_t kTmemCols = QB ? kMxTmemCols : kSkTmemCols;
    if (warp == 1) {
        tmem_alloc(slot_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot_ptr;

    // fp16 B: the operand ring (B^T + A per stage).  QB: the raw ring (codes +
    // scales + A).
    constexpr int kRing = QB ? kRaw : kSkStages;
    constexpr int kProd = skinny_producers(kRing);
    static_assert(kRing % kProd == 0, "each ring stage must belong to one producer thread");
    constexpr int kMma2Warp = QB ? 6 + kMxConvWarps : -1;  // QB: the second MMA warp
    constexpr int kProdWarp1 = 6 + (QB ? kMxConvWarps + 1 : 0);  // warp of producer 1
    constexpr int kAProdWarp = QB ? kProdWarp1 + kProd - 1 : -1;  // QB: A ring producer
    const int prod = warp == 0 ? 0
                     : (warp >= kProdWarp1 && warp < kProdWarp1 + kProd - 1 ? warp - kProdWarp1 + 1
                                                                             : -1);
    // Producer set-up that reads no data of the previous kernel (cache
    // policies, the first unit's tile and k block: a 64-bit division) is done
    // before the dependency wait.
    uint64_t keep_policy = 0, stream_policy = 0;
    int32_t prod_t = 0, prod_kb = 0;  // producer thread: (tile, k block) of its first unit
    int32_t a_kb = 0;                 // QB, A ring producer: its first k block
    if (lane == 0 && (prod >= 0 || warp == kAProdWarp)) {
        keep_policy = policy_evict_last();     // A: reread by every CTA
        stream_policy = policy_evict_first();  // B: read exactly once
        if (prod >= 0) {
            const int64_t u0 = u_begin + prod;
            prod_t = static_cast<int32_t>(u0 / KB);
            prod_kb = static_cast<int32_t>(u0 - static_cast<int64_t>(prod_t) * KB);
        } else {
            a_kb = static_cast<int32_t>(u_begin % KB);
        }
    }
    if (warp == 0 && lane == 0) {
        // the first ring's worth of this CTA's units into L2 while the
        // previous kernel finishes (producer 0's first unit is u_begin)
        int32_t t = prod_t;
        int32_t kb = prod_kb;
        // (MXFP4: two units.  Prefetching the whole raw ring kept the TMA unit
        // busy for about 3 us after the dependency wait, and the first loads
        // queued behind it.)
        constexpr int kAhead = QB ? 2 : kSkStages;
        for (int i = 0; i < kAhead && u_begin + i < u_end; ++i) {
            if constexpr (QB) {
#pragma unroll
                for (int h = 0; h < BK / 64; ++h)
                    tma_prefetch_2d(tmB, kb * (BK / 2) + 32 * h, t * 128);
                tma_prefetch_2d(tmS, t * 128, kb * (BK / 32));
            } else {
                tma_prefetch_2d(tmB, t * 128, kb * BK);
                tma_prefetch_2d(tmB, t * 128 + 64, kb * BK);
            }
#pragma unroll
            for (int h = 0; h < BK / 64; ++h) tma_prefetch_2d(tmA, kb * BK + 64 * h, 0);
            if (++kb == static_cast<int32_t>(KB)) {
                kb = 0;
                ++t;
            }
        }
    }
    grid_dependency_wait();  // the previous kernel's writes are visible from here on
    grid_launch_dependents();

    auto fail = [&](unsigned int role) {
        atomicOr(&g_wait_timeout_flags, role);
        *abort_flag = 1;
    };

    if (prod >= 0) {
        // ------------------------------------------------------------ producers
        if (lane == 0) {
            const uint64_t keep = keep_policy;
            const uint64_t stream = stream_policy;
            const uint32_t ring_full = QB ? bar_rfull : bar_full;
            const uint32_t ring_empty = QB ? bar_rempty : bar_empty;
            uint32_t issued_mask = 0, issued_parity = 0;
            // (tile, k block) of this producer's next unit, advanced by kProd
            // units per step (no division per unit)
            int32_t t = prod_t;
            int32_t kb = prod_kb;
            for (int64_t i = prod; u_begin + i < u_end; i += kProd) {
                const int stage = static_cast<int>(i % kRing);
                const uint32_t phase = static_cast<uint32_t>((i / kRing) & 1);
                if (!mbar_wait(ring_empty + 8 * stage, phase ^ 1u, p.timeout_ns, abort_flag)) {
                    fail(kRoleProducer);
                    break;
                }
                const uint32_t full = ring_full + 8 * stage;
                if constexpr (QB) {
                    mbar_arrive_expect_tx(full, kMxRawBytes + kMxScaleBytes);
#pragma unroll
                    for (int h = 0; h < BK / 64; ++h)  // codes: BK / 2 bytes of k per column
                        tma_load_2d_hint(sRaw + stage * kMxRawBytes + kMxCodeBox * h, tmB, full,
                                         kb * (BK / 2) + 32 * h, t * 128, stream);
                    tma_load_2d_hint(sScl + stage * kMxScaleBytes, tmS, full, t * 128,
                                     kb * (BK / 32), stream);
                } else {
                    mbar_arrive_expect_tx(full, kSkBBytes + (BK / 64) * a_bytes);
                    const uint32_t b0 = sB + stage * kSkBBytes;
                    tma_load_2d_hint(b0, tmB, full, t * 128, kb * BK, stream);
                    tma_load_2d_hint(b0 + kSkBBytes / 2, tmB, full, t * 128 + 64, kb * BK, stream);
#pragma unroll
                    for (int i = 0; i < BK / 64; ++i)
                        tma_load_2d_hint(sA + stage * kSkASlot + kABox * i, tmA, full,
                                         kb * BK + 64 * i, 0, keep);
                }
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                kb += kProd;
                while (kb >= KB) {
                    kb -= static_cast<int32_t>(KB);
                    ++t;
                }
            }
            for (int s = 0; s < kRing; ++s)
                if (issued_mask & (1u << s))
                    if (!mbar_wait(ring_full + 8 * s, (issued_parity >> s) & 1u, p.timeout_ns,
                                   nullptr))
                        atomicOr(&g_wait_timeout_flags, kRoleDrain);
        }
    } else if (warp == kAProdWarp) {
        // ------------------------------------------------------------ A ring producer (QB)
        if constexpr (QB) if (lane == 0) {
            const uint64_t keep = keep_policy;
            uint32_t issued_mask = 0, issued_parity = 0;
            int32_t kb = a_kb;
            for (int64_t i = 0; u_begin + i < u_end; ++i) {
                const int stage = static_cast<int>(i % kAS);
                const uint32_t phase = static_cast<uint32_t>((i / kAS) & 1);
                // the MMAs of the unit kAS earlier (same A stage) are done
                if (!mbar_wait(bar_aempty + 8 * stage, phase ^ 1u, p.timeout_ns, abort_flag)) {
                    fail(kRoleProducer);
                    break;
                }
                const uint32_t full = bar_afull + 8 * stage;
                mbar_arrive_expect_tx(full, (BK / 64) * a_bytes);
#pragma unroll
                for (int h = 0; h < BK / 64; ++h)
                    tma_load_2d_hint(sA + stage * kSkASlot + kABox * h, tmA, full,
                                     kb * BK + 64 * h, 0, keep);
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++kb == KB) kb = 0;
            }
            for (int a = 0; a < kAS; ++a)
                if (issued_mask & (1u << a))
                    if (!mbar_wait(bar_afull + 8 * a, (issued_parity >> a) & 1u, p.timeout_ns,
                                   nullptr))
                        atomicOr(&g_wait_timeout_flags, kRoleDrain);
        }
    } else if (warp == 1 || warp == kMma2Warp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (warp-uniform control flow and
        // operands); one elected lane issues each MMA and commit.  A wait
        // counts as met only if every lane saw it met.  QB: MMA warp m takes
        // the units u + m, u + m + kMW, ... of each segment [u, seg_end).
        auto warp_wait = [&](uint32_t bar, uint32_t parity, const volatile int* ab) {
            const bool r = mbar_wait(bar, parity, p.timeout_ns, ab);
            return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
        };
        const int m = warp == 1 ? 0 : 1;
        // fp16 B: A operand = B^T tile, MN-major in shared memory.  QB: A
        // operand = decoded weights in tensor memory (K-major).
        const uint32_t idesc =
            idesc_f16_f32(128, p.Mp, /*a_mn=*/!QB, /*b_mn=*/false, Elem16<T>::kFmt);
        int it = 0;
        bool ok = true;
        for (int64_t u = u_begin; ok && u < u_end; ++it) {
            const int64_t t = u / KB;
            const int64_t seg_end = (t + 1) * KB < u_end ? (t + 1) * KB : u_end;
            const int buf = it % kBufs;
            const uint32_t buf_phase = static_cast<uint32_t>((it / kBufs) & 1);
            if (!warp_wait(bar_tempty + 8 * buf, buf_phase ^ 1u, abort_flag)) {
                if (lane == 0) fail(kRoleMma);
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem =
                tmem_base + static_cast<uint32_t>(buf * kMW + m) * kAccStride;
            for (int64_t v = u + m; v < seg_end; v += kMW) {
                const int64_t i = v - u_begin;  // local unit index
                const int stage = static_cast<int>(i % kSkStages);
                const uint32_t phase = static_cast<uint32_t>((i / kSkStages) & 1);
                // QB: B^T decoded into the operand stage, and (the
                // converters waited for it) the unit's A tile landed
                const bool got = warp_wait(QB ? bar_dec + 8 * stage : bar_full + 8 * stage,
                                           phase, abort_flag);
                if (!got) {
                    if (lane == 0) fail(kRoleMma);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                if constexpr (QB) {
                    static_assert(BK == 128, "the unit issue below covers 128 k");
                    const int astage = static_cast<int>(i % kAS);
                    mx_unit_mma_elect<kABox / 16>(
                        d_tmem, tmem_base + kOpCol0 + static_cast<uint32_t>(kMxOpCols * stage),
                        smem_desc_sw128(sA + astage * kSkASlot, 16, 1024), idesc,
                        v - u < kMW ? 1u : 0u, bar_empty + 8 * stage, bar_aempty + 8 * astage);
                } else {
                    const uint32_t b0 = sB + stage * kSkBBytes;
                    const uint32_t a0 = sA + stage * kSkASlot;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // A tile: 64-k boxes kABox apart, 32 B per 16 k inside one
                        const uint64_t bdesc =
                            smem_desc_sw128(a0 + kABox * (k / 4) + 32 * (k % 4), 16, 1024);
                        const uint32_t acc_in = (v != u || k != 0) ? 1u : 0u;
                        // B^T: 16 k rows (2 KB) per step; the two 64-column boxes
                        // kSkBBytes / 2 apart
                        const uint64_t adesc =
                            smem_desc_sw128(b0 + 2048 * k, kSkBBytes / 2, 1024);
                        mma_f16_ss_elect(d_tmem, adesc, bdesc, idesc, acc_in);
                    }
                    mma_commit_elect(bar_empty + 8 * stage);
                }
            }
            if (!ok) break;
            if (!(p.inject == 1 && it == 0)) mma_commit_elect(bar_tfull + 8 * buf);
            u = seg_end;
        }
        mma_commit_elect(bar_drain);
        if (!warp_wait(bar_drain, 0, nullptr) && lane == 0)
            atomicOr(&g_wait_timeout_flags, kRoleDrain);
    } else if (warp >= 2 && warp < 6) {
        // ------------------------------------------------------------ epilogue
        // The parameters it uses, in registers: read through the parameter
        // reference, every store to C (which the compiler cannot prove
        // apart from them) forced them to be read again, and a tile's
        // epilogue took about 7000 cycles.
        const int Mr = p.M, Nr = p.N, Mp = p.Mp, relu = p.relu, out_f32 = p.out_f32;
        const int64_t ldc = p.ldc, ldr = p.e.ldr;
        void* const Cv = p.C;
        const float* const bias = p.e.bias;
        const void* const resid = p.e.resid;
        float* const ws = p.ws;
        uint32_t* const counters = p.counters;
        const uint64_t timeout_ns = p.timeout_ns;
        const int q = warp & 3;
        const int n_local = 32 * q + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        int it = 0;
        for (int64_t u = u_begin; u < u_end; ++it) {
            const int64_t t = u / KB;
            const int64_t kb0 = u - t * KB;
            const int64_t seg_end = (t + 1) * KB < u_end ? (t + 1) * KB : u_end;
            const int64_t kb1 = seg_end - t * KB;
            const int acc = it % kBufs;
            const uint32_t acc_phase = static_cast<uint32_t>((it / kBufs) & 1);
            const int64_t n = t * 128 + n_local;
            int ok = 1;
            if (lane == 0)
                ok = mbar_wait(bar_tfull + 8 * acc, acc_phase, timeout_ns, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) fail(kRoleEpilogue);
                break;
            }
            tc_fence_after_sync();
            const uint32_t tacc =
                tmem_base + lane_addr + static_cast<uint32_t>(acc * kMW) * kAccStride;
            // QB: the second MMA warp's accumulator holds units iff the
            // segment has two or more
            const bool two = kMW > 1 && seg_end - u >= 2;
            // Chunk c (32 m) of this thread's column: the accumulators' sum, in
            // one tensor-memory round trip.  Rows past Mp read columns that
            // are not this accumulator's (garbage, never stored).  A round
            // trip per 16 m made the epilogue of a tile take about 7000 cycles.
            // (With two accumulators the chunks are 16 m: 32 registers per
            // load pair, within the MXFP4 kernel's register budget.)
            constexpr int CW = kMW > 1 ? 16 : 32;
            static_assert(kAccStride >= CW, "chunks stay inside the allocation");
            auto load_acc = [&](int c, uint32_t (&r)[CW]) {
                if constexpr (CW == 16) {
                    if (two) {
                        uint32_t r2[16];
                        tmem_ld2_x16(tacc + 16 * c, tacc + kAccStride + 16 * c, r, r2);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
                    } else {
                        tmem_ld_x16(tacc + 16 * c, r);
                    }
                } else {
                    tmem_ld_x32(tacc + 32 * c, r);
                }
            };
            const int nchunksw = (Mp + CW - 1) / CW;

            // The slots this warp sums, in k order (none: a FULL segment,
            // summed from tensor memory alone).
            int64_t c_head = 0, c_last = -1;
            if (kb0 > 0 || kb1 < KB) {
                // A piece of a split tile: its fp32 partial to this CTA's
                // slot for it, layout [m][n_local].
                const int64_t my_slot = 2 * static_cast<int64_t>(blockIdx.x) + (kb0 > 0 ? 0 : 1);
                float* slot = ws + my_slot * kSkSlotFloats;
                for (int c = 0; c < nchunksw; ++c) {
                    uint32_t r[CW];
                    load_acc(c, r);
#pragma unroll
                    for (int i = 0; i < CW; ++i)
                        if (CW * c + i < Mp)
                            __stcg(slot + (CW * c + i) * 128 + n_local, __uint_as_float(r[i]));
                }
                tc_fence_before_sync();
                __threadfence();
                __syncwarp();
                // The accumulator is free.  Count this piece in; the warp
                // that brings the count to the tile's number of pieces sums
                // them all.
                c_head = unit_owner(t * KB, G, U);
                const int64_t c_tail = unit_owner((t + 1) * KB - 1, G, U);
                int last = 0;
                if (lane == 0) {
                    mbar_arrive(bar_tempty + 8 * acc);
                    uint32_t* cnt = counters + 4 * c_head + q;
                    const uint32_t before = atomic_add_acq_rel_gpu(cnt, 1u);
                    last = before + 1 == static_cast<uint32_t>(c_tail - c_head + 1) ? 1 : 0;
                    if (last) *cnt = 0u;  // zero again for the next launch
                }
                if (!__shfl_sync(0xffffffffu, last, 0)) {
                    u = seg_end;
                    continue;
                }
                __threadfence();
                c_last = c_tail;
            }
            // FULL, or the last piece of a split tile in: C[m][n] =
            // out(act(sum + bias[n]) + R[m][n]); this thread holds column n.
            for (int c = 0; c < nchunksw; ++c) {
                float v[CW];
                if (c_last < 0) {
                    uint32_t r[CW];
                    load_acc(c, r);
#pragma unroll
                    for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]);
                } else {
                    // the head's piece (its second slot), then the first
                    // pieces of CTAs c_head + 1 .. c_last: k order
                    const float* h = ws + (2 * c_head + 1) * kSkSlotFloats;
#pragma unroll
                    for (int i = 0; i < CW; ++i)
                        v[i] = CW * c + i < Mp ? __ldcg(h + (CW * c + i) * 128 + n_local) : 0.0f;
                    for (int64_t cc = c_head + 1; cc <= c_last; ++cc) {
                        const float* slot = ws + 2 * cc * kSkSlotFloats;
#pragma unroll
                        for (int i = 0; i < CW; ++i)
                            if (CW * c + i < Mp) v[i] += __ldcg(slot + (CW * c + i) * 128 + n_local);
                    }
                }
                if constexpr (!EX) {
                    // Plain build: one row per step through a pointer.  (The
                    // general body below, with its per-element branches and
                    // offsets, is a few KB of code run once per chunk: it took
                    // about 1500 cycles per chunk, with or without its loads
                    // and stores.)
                    if (n < Nr) {
                        T* cp = static_cast<T*>(Cv) + static_cast<int64_t>(CW * c) * ldc + n;
                        const int rows = Mr - CW * c;  // rows of this chunk inside C
#pragma unroll
                        for (int i = 0; i < CW; ++i) {
                            float x = v[i];
                            if (relu) x = relu_f32(x);
                            if (i < rows) *cp = Elem16<T>::from_float(x);
                            cp += ldc;
                        }
                    }
                } else if (n < Nr) {
                    const float bias_n = bias != nullptr ? __ldg(bias + n) : 0.0f;
#pragma unroll
                    for (int i = 0; i < CW; ++i) {
                        const int m = CW * c + i;
                        if (m < Mr) {
                            float x = v[i];
                            if (bias != nullptr) x += bias_n;
                            if (relu) x = relu_f32(x);
                            if (resid != nullptr)
                                x += Elem16<T>::to_float(
                                    static_cast<const T*>(resid)[static_cast<int64_t>(m) * ldr + n]);
                            const int64_t off = static_cast<int64_t>(m) * ldc + n;
                            if (out_f32)
                                static_cast<float*>(Cv)[off] = x;
                            else
                                static_cast<T*>(Cv)[off] = Elem16<T>::from_float(x);
                        }
                    }
                }
            }
            if (c_last < 0) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
            }
            u = seg_end;
        }
    } else if constexpr (QB) {
        // ------------------------------------------------------------ converters (QB)
        // (warps 6 .. 6 + kMxConvWarps - 1)
        // Warp cw = warp - 6 is in group g = cw / kMxGroupWarps, owns
        // tensor-memory lane quarter q = warp % 4 and decodes half hh =
        // (cw % kMxGroupWarps) / 4 (k 64 hh .. 64 hh + 63) of each unit of
        // local index i ≡ g (mod kMxGroups): thread l decodes column n = 32 q
        // + l, its 64 k codes (32 bytes: row n of the codes tile, 32-byte
        // swizzle) with the half's two block scales, into 32 columns of fp16
        // pairs (lower k in the low half), stored to its lane of the unit's
        // operand stage.
        const int cw = warp - 6;
        const int g = cw / kMxGroupWarps;
        const uint32_t hh0 = static_cast<uint32_t>((cw % kMxGroupWarps) / 4 * kMxHalvesPerWarp);
        const uint32_t q = static_cast<uint32_t>(warp & 3);
        const uint32_t n_local = 32u * q + static_cast<uint32_t>(lane);
        const uint32_t swz32 = (n_local >> 2) & 1u;
        const uint32_t lane_addr = (32u * q) << 16;
        static_assert(BK == 128 || !QB, "two 64-k halves per unit");
        for (int64_t i = g; u_begin + i < u_end; i += kMxGroups) {
            const int stage = static_cast<int>(i % kSkStages);
            const uint32_t phase = static_cast<uint32_t>((i / kSkStages) & 1);
            const int rstage = static_cast<int>(i % kRaw);
            const uint32_t rphase = static_cast<uint32_t>((i / kRaw) & 1);
            int ok = 1;
            if (lane == 0) {
                // the MMAs that read this operand stage have completed, and
                // the unit's codes have landed
                ok = mbar_wait(bar_empty + 8 * stage, phase ^ 1u, p.timeout_ns, abort_flag) ? 1
                                                                                            : 0;
                if (ok)
                    ok = mbar_wait(bar_rfull + 8 * rstage, rphase, p.timeout_ns, abort_flag) ? 1
                                                                                             : 0;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) fail(kRoleConvert);
                break;
            }
            tc_fence_after_sync();
            // This half's codes and scales into registers, then the raw
            // stage is free for the next load (once the group's warps all
            // have theirs).
            uint32_t w[kMxHalvesPerWarp][8];
            uint32_t X0[kMxHalvesPerWarp], X1[kMxHalvesPerWarp];
#pragma unroll
            for (int h = 0; h < kMxHalvesPerWarp; ++h) {
                const uint32_t hh = hh0 + static_cast<uint32_t>(h);
                const uint32_t row = sRaw + static_cast<uint32_t>(rstage) * kMxRawBytes +
                                     kMxCodeBox * hh + 32u * n_local;
                const uint4 c0 = mx_ld_shared_v4(row + (swz32 << 4));
                const uint4 c1 = mx_ld_shared_v4(row + ((swz32 ^ 1u) << 4));
                const uint32_t scl = sScl + static_cast<uint32_t>(rstage) * kMxScaleBytes +
                                     256u * hh + n_local;
                X0[h] = mx_ld_shared_u8(scl);
                X1[h] = mx_ld_shared_u8(scl + 128u);
                w[h][0] = c0.x;
                w[h][1] = c0.y;
                w[h][2] = c0.z;
                w[h][3] = c0.w;
                w[h][4] = c1.x;
                w[h][5] = c1.y;
                w[h][6] = c1.z;
                w[h][7] = c1.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_rempty + 8 * rstage);
#pragma unroll
            for (int h = 0; h < kMxHalvesPerWarp; ++h) {
                const uint32_t hh = hh0 + static_cast<uint32_t>(h);
                uint32_t d[32];
                if (mx_fast_scale(X0[h]) && mx_fast_scale(X1[h])) {
                    const uint32_t f0 = mx_factor_bits(X0[h]) * 0x10001u;  // both halves
                    const uint32_t f1 = mx_factor_bits(X1[h]) * 0x10001u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t f = j < 4 ? f0 : f1;  // words 0..3: k 0..31
                        const uint32_t fj[4] = {f, f, f, f};
                        const uint4 o = mx_decode8_fast(w[h][j], fj);
                        d[4 * j] = o.x;
                        d[4 * j + 1] = o.y;
                        d[4 * j + 2] = o.z;
                        d[4 * j + 3] = o.w;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t xb = j < 4 ? X0[h] : X1[h];
                        const uint32_t x[8] = {xb, xb, xb, xb, xb, xb, xb, xb};
                        const uint4 o = mx_decode8_exact(w[h][j], x);
                        d[4 * j] = o.x;
                        d[4 * j + 1] = o.y;
                        d[4 * j + 2] = o.z;
                        d[4 * j + 3] = o.w;
                    }
                }
                __syncwarp();
                mx_tmem_st_x32(tmem_base + lane_addr + kOpCol0 +
                                   static_cast<uint32_t>(kMxOpCols * stage) + 32u * hh,
                               d);
            }
            mx_tmem_wait_st();
            // the unit's A tile (its load overlapped the decode): the MMA
            // warp then waits on one barrier per unit
            if (lane == 0)
                ok = mbar_wait(bar_afull + 8 * static_cast<int>(i % kAS),
                               static_cast<uint32_t>((i / kAS) & 1), p.timeout_ns, abort_flag)
                         ? 1
                         : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) fail(kRoleConvert);
                break;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_dec + 8 * stage);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int STAGES, int MP_MAX, typename T = __half, int BK = 64, bool EX = true>
__global__ void __launch_bounds__(skinny_threads(STAGES, MP_MAX, false), 1)
    tg_gemm_f16_skinny(const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmA, const SkinnyParams p) {
    skinny_body<STAGES, MP_MAX, T, false, BK, EX>(&tmB, &tmA, nullptr, p);
}

// C = epi(A · Bdeq) with B in MXFP4 (mxfp4.cuh), M ≤ 128, A fp16.
template <int STAGES, int MP_MAX, bool EX = true>
__global__ void __launch_bounds__(skinny_threads(STAGES, MP_MAX, true), 1)
    tg_gemm_mxfp4_skinny(const __grid_constant__ CUtensorMap tmBq,
                         const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmS, const SkinnyParams p) {
    skinny_body<STAGES, MP_MAX, __half, true, kMxBK, EX>(&tmBq, &tmA, &tmS, p);
}

// ------------------------------------------------------------------ host side

inline bool skinny_applies(int64_t M, int64_t N, int64_t K) {
    (void)N;
    (void)K;
    return M >= 1 && M <= 128;
}

// A grid that cuts the units only at tile edges or at equal fractions of a
// tile: T / d CTAs of d whole tiles each (d divides T), or T · s CTAs of one
// 1/s k-range each, whichever is closer to num_sms; 0 if neither reaches
// 0.7 num_sms or would give a CTA fewer than kSkMinUnitsPerCta units.  Each
// CTA then streams whole tiles (no partial sums) or one equal piece of one.
inline int64_t skinny_aligned_grid(int64_t T, int64_t KB, int32_t num_sms) {
    int64_t best = 0;
    for (int64_t d = 1; d <= T; ++d)
        if (T % d == 0 && T / d <= num_sms) {
            best = T / d;
            break;
        }
    const int64_t s = T > 0 ? num_sms / T : 0;
    if (s >= 2 && KB / s >= kSkMinUnitsPerCta && T * s > best) best = T * s;
    if (10 * best < 7 * static_cast<int64_t>(num_sms)) return 0;
    if (T * KB / best < kSkMinUnitsPerCta) return 0;
    return best;
}

// Units of bk k (the fp16/bf16 kernel: SkinnyNarrow/Wide::kBK; MXFP4: kMxBK).
// align: take skinny_aligned_grid when it applies.  The fp16/bf16 kernel is
// bound by streaming B, and on 64×16384×8192 one CTA per whole tile (128
// CTAs) measured 43.0 µs against 48.8 µs for 152 CTAs with pieces; on
// 128×28672×4096 two whole tiles per CTA (112 CTAs) 47.0 against 53.4 µs.
// The MXFP4 kernel takes it too: on 64×16384×8192 one CTA per tile measured
// 30.1 µs against 33.6 µs for 152 CTAs with pieces and their fix-up.
inline void skinny_plan_bk(int64_t M, int64_t N, int64_t K, int32_t num_sms, int32_t bk,
                           tg_plan_t* pl, bool align = false) {
    const int64_t Mp = (M + 15) / 16 * 16;
    const bool narrow = Mp <= 64;
    pl->kernel = TG_KERNEL_SKINNY;
    pl->bm = static_cast<int32_t>(Mp);
    pl->bn = 128;
    pl->bk = bk;
    pl->stages = narrow ? SkinnyNarrow::kStages : SkinnyWide::kStages;
    pl->mma_m = 128;
    pl->mma_n = static_cast<int32_t>(Mp);
    pl->tiles_m = 1;
    pl->tiles_n = (N + 127) / 128;
    pl->k_blocks = (K + bk - 1) / bk;
    pl->num_tiles = pl->tiles_n;
    const int64_t U = pl->tiles_n * pl->k_blocks;
    int64_t G = U / kSkMinUnitsPerCta;
    if (G < 1) G = 1;
    if (G > num_sms) G = num_sms;
    int64_t aligned = 0;
    if (align) {
        aligned = skinny_aligned_grid(pl->tiles_n, pl->k_blocks, num_sms);
        if (aligned > 0) G = aligned;
    }
    pl->grid = G;
    pl->threads = narrow ? skinny_threads(SkinnyNarrow::kStages, 64, false)
                         : skinny_threads(SkinnyWide::kStages, 128, false);
    pl->group_m = 1;
    pl->smem_bytes = narrow ? SkinnyNarrow::kSmemBytes : SkinnyWide::kSmemBytes;
    pl->ring_bytes = narrow ? int64_t{SkinnyNarrow::kStages} * SkinnyNarrow::kStageBytes
                            : int64_t{SkinnyWide::kStages} * SkinnyWide::kStageBytes;
    // most CTAs touching one tile: exact for an aligned grid; else its k range
    // over the shortest unit range, plus one
    const int64_t shortest = U / G;
    if (aligned > 0)
        pl->split_k = G <= pl->tiles_n ? 1 : G / pl->tiles_n;
    else
        pl->split_k = shortest > 0 ? (pl->k_blocks + shortest - 1) / shortest + 1 : pl->k_blocks;
    if (pl->split_k > G) pl->split_k = G;
    pl->workspace_bytes = 2 * G * kSkSlotFloats * 4 + 4 * G * 4;
    // Four k-pieces per tile (G = 4 T): the launch groups each tile's four
    // CTAs into one cluster.  Back to back on one box: 64×4096×4096 17.3 ->
    // 16.1 µs, 128×4096×14336 37.1 -> 33.8 µs, 32×4096×14336 24.8 -> 24.2 µs,
    // M = 1 and 16 unchanged.  Whole-tile grids took 0.5 % longer that way and
    // 2 or 3 pieces per tile gained nothing, so they launch without clusters.
    // The launch drops the clusters if not all of them fit on the device at
    // once (a second round of clusters would double the time).
    pl->cluster = (aligned > 0 && G == 4 * pl->tiles_n) ? 4 : 1;
}

inline void skinny_plan(int64_t M, int64_t N, int64_t K, int32_t num_sms, tg_plan_t* pl) {
    const bool narrow = (M + 15) / 16 * 16 <= 64;
    skinny_plan_bk(M, N, K, num_sms, narrow ? SkinnyNarrow::kBK : SkinnyWide::kBK, pl, true);
}

// The MXFP4 kernel: the same units and split, its own rings and 448 threads.
inline void skinny_mx_plan(int64_t M, int64_t N, int64_t K, int32_t num_sms, tg_plan_t* pl) {
    skinny_plan_bk(M, N, K, num_sms, kMxBK, pl, true);
    pl->cluster = 1;  // the MXFP4 kernel launches without clusters
    const bool narrow = pl->bm <= 64;
    pl->stages = narrow ? SkinnyMxNarrow::kStages : SkinnyMxWide::kStages;
    pl->threads = narrow ? skinny_threads(SkinnyMxNarrow::kStages, 64, true)
                         : skinny_threads(SkinnyMxWide::kStages, 128, true);
    pl->smem_bytes = narrow ? SkinnyMxNarrow::kSmemBytes : SkinnyMxWide::kSmemBytes;
    pl->ring_bytes =
        narrow ? int64_t{SkinnyMxNarrow::kRawStages} * SkinnyMxNarrow::kRawStageBytes +
                     int64_t{SkinnyMxNarrow::kAStages} * SkinnyMxNarrow::kASlot
               : int64_t{SkinnyMxWide::kRawStages} * SkinnyMxWide::kRawStageBytes +
                     int64_t{SkinnyMxWide::kAStages} * SkinnyMxWide::kASlot;
}

template <bool EX>
inline cudaError_t skinny_mx_set_attributes_ex() {
    cudaError_t e = cudaFuncSetAttribute(tg_gemm_mxfp4_skinny<SkinnyMxNarrow::kStages, 64, EX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SkinnyMxNarrow::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(tg_gemm_mxfp4_skinny<SkinnyMxWide::kStages, 128, EX>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SkinnyMxWide::kSmemBytes);
}

inline cudaError_t skinny_mx_set_attributes() {
    const cudaError_t e = skinny_mx_set_attributes_ex<true>();
    return e != cudaSuccess ? e : skinny_mx_set_attributes_ex<false>();
}

template <typename T, bool EX>
inline cudaError_t skinny_set_attributes_ex() {
    cudaError_t e = cudaFuncSetAttribute(
        tg_gemm_f16_skinny<SkinnyNarrow::kStages, 64, T, SkinnyNarrow::kBK, EX>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, SkinnyNarrow::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(
        tg_gemm_f16_skinny<SkinnyWide::kStages, 128, T, SkinnyWide::kBK, EX>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, SkinnyWide::kSmemBytes);
}

template <typename T>
inline cudaError_t skinny_set_attributes() {
    const cudaError_t e = skinny_set_attributes_ex<T, true>();
    return e != cudaSuccess ? e : skinny_set_attributes_ex<T, false>();
}

// The plain-epilogue build applies: no bias, no residual, 16-bit C.
inline bool skinny_plain(const SkinnyParams& prm) {
    return prm.e.bias == nullptr && prm.e.resid == nullptr && prm.out_f32 == 0;
}

// Launch of the instantiation whose A slots fit prm.Mp.
template <typename T>
inline cudaError_t skinny_launch_kernel(const CUtensorMap& tmB, const CUtensorMap& tmA,
                                        const SkinnyParams& prm, int64_t grid,
                                        cudaStream_t stream, int32_t cluster = 1) {
    cudaLaunchAttribute attr[2];
    set_dependent_launch(attr[0]);
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(prm.Mp <= 64 ? skinny_threads(SkinnyNarrow::kStages, 64, false)
                                     : skinny_threads(SkinnyWide::kStages, 128, false));
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 && grid % cluster == 0 ? 2 : 1;
    using N = SkinnyNarrow;
    using Wd = SkinnyWide;
    const bool plain = skinny_plain(prm);
    if (prm.Mp <= 64) {
        cfg.dynamicSmemBytes = N::kSmemBytes;
        return plain ? cudaLaunchKernelEx(&cfg,
                                          tg_gemm_f16_skinny<N::kStages, 64, T, N::kBK, false>,
                                          tmB, tmA, prm)
                     : cudaLaunchKernelEx(&cfg, tg_gemm_f16_skinny<N::kStages, 64, T, N::kBK>, tmB,
                                          tmA, prm);
    }
    cfg.dynamicSmemBytes = Wd::kSmemBytes;
    return plain ? cudaLaunchKernelEx(&cfg, tg_gemm_f16_skinny<Wd::kStages, 128, T, Wd::kBK, false>,
                                      tmB, tmA, prm)
                 : cudaLaunchKernelEx(&cfg, tg_gemm_f16_skinny<Wd::kStages, 128, T, Wd::kBK>, tmB,
                                      tmA, prm);
}

// Launch of the MXFP4 instantiation whose A slots fit prm.Mp.
inline cudaError_t skinny_mx_launch_kernel(const CUtensorMap& tmBq, const CUtensorMap& tmA,
                                           const CUtensorMap& tmS, const SkinnyParams& prm,
                                           int64_t grid, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    set_dependent_launch(attr[0]);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(prm.Mp <= 64 ? skinny_threads(SkinnyMxNarrow::kStages, 64, true)
                                     : skinny_threads(SkinnyMxWide::kStages, 128, true));
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool plain = skinny_plain(prm);
    if (prm.Mp <= 64) {
        cfg.dynamicSmemBytes = SkinnyMxNarrow::kSmemBytes;
        return plain ? cudaLaunchKernelEx(&cfg,
                                          tg_gemm_mxfp4_skinny<SkinnyMxNarrow::kStages, 64, false>,
                                          tmBq, tmA, tmS, prm)
                     : cudaLaunchKernelEx(&cfg, tg_gemm_mxfp4_skinny<SkinnyMxNarrow::kStages, 64>,
                                          tmBq, tmA, tmS, prm);
    }
    cfg.dynamicSmemBytes = SkinnyMxWide::kSmemBytes;
    return plain ? cudaLaunchKernelEx(&cfg, tg_gemm_mxfp4_skinny<SkinnyMxWide::kStages, 128, false>,
                                      tmBq, tmA, tmS, prm)
                 : cudaLaunchKernelEx(&cfg, tg_gemm_mxfp4_skinny<SkinnyMxWide::kStages, 128>, tmBq,
                                      tmA, tmS, prm);
}

struct SplitkWorkspace {
    float* partials = nullptr;    // two slots per CTA
    uint32_t* counters = nullptr;  // four per CTA
    int64_t ctas = 0;
};

inline std::mutex& splitk_ws_mutex() {
    static std::mutex m;
    return m;
}

inline std::map<std::pair<int, cudaStream_t>, SplitkWorkspace>& splitk_ws_map() {
    static std::map<std::pair<int, cudaStream_t>, SplitkWorkspace> m;
    return m;
}

// After a launch gave up on a wait, some tiles' counters may never have
// reached their piece count (and been zeroed): reset every workspace's
// counters on this device (the device is idle).
inline void splitk_reset_counters(int dev) {
    std::lock_guard<std::mutex> lk(splitk_ws_mutex());
    for (auto& kv : splitk_ws_map())
        if (kv.first.first == dev && kv.second.counters != nullptr)
            cudaMemset(kv.second.counters, 0, 4 * kv.second.ctas * sizeof(uint32_t));
}

// The split-K workspace of (dev, stream) into prm (ws, counters); sized on
// first use for the largest grid, so later calls never grow it.  The pair
// kernel's split tail tiles use it too (one 256 KB slot per cluster, eight
// counters per tail tile: within the same bytes for a grid of one CTA per
// SM); launches on one stream are ordered, so they never share it at once.
inline tg_status_t splitk_workspace(int dev, cudaStream_t stream, int64_t grid, int64_t max_ctas,
                                    SkinnyParams* prm) {
    {
        std::lock_guard<std::mutex> lk(splitk_ws_mutex());
        SplitkWorkspace& ws = splitk_ws_map()[std::make_pair(dev, stream)];
        if (ws.ctas < grid) {
            // First use on this stream: room for the largest grid (one CTA
            // per SM), so later calls, graph captures included, never grow it.
            if (ws.partials) {
                cudaStreamSynchronize(stream);
                cudaFree(ws.partials);
                cudaFree(ws.counters);
                ws.partials = nullptr;
                ws.counters = nullptr;
                ws.ctas = 0;
            }
            const int64_t ctas = grid > max_ctas ? grid : max_ctas;
            if (cudaMalloc(&ws.partials, 2 * ctas * kSkSlotFloats * sizeof(float)) !=
                    cudaSuccess ||
                cudaMalloc(&ws.counters, 4 * ctas * sizeof(uint32_t)) != cudaSuccess) {
                cudaGetLastError();
                if (ws.partials) cudaFree(ws.partials);
                ws.partials = nullptr;
                ws.counters = nullptr;
                return TG_ERR_NO_MEMORY;
            }
            if (cudaMemsetAsync(ws.counters, 0, 4 * ctas * sizeof(uint32_t), stream) !=
                cudaSuccess) {
                cudaGetLastError();
                return TG_ERR_LAUNCH;
            }
            ws.ctas = ctas;
        }
        prm->ws = ws.partials;
        prm->counters = ws.counters;  // zero between launches (the last piece zeroes them)
    }
    return TG_OK;
}

using EncodeFn = bool (*)(CUtensorMap*, const void*, uint64_t, uint64_t, uint64_t, uint32_t,
                          uint32_t, CUtensorMapDataType);

template <typename T>
inline tg_status_t skinny_launch(const void* A, const void* B, void* C, const tg_plan_t& pl,
                                 int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                 int64_t ldc, const EpilogueSpec& ep, cudaStream_t stream, int dev,
                                 int64_t max_ctas, uint64_t timeout_ns, int32_t inject,
                                 EncodeFn encode) {
    const int64_t Mp = pl.mma_n;
    CUtensorMap tmA, tmB;
    const CUtensorMapDataType dt = Elem16<T>::kFmt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // B: boxes of 64 columns × (the unit's k) rows; A: 64-k boxes of Mp rows
    if (!encode(&tmB, B, N, K, ldb * 2, 64, static_cast<uint32_t>(pl.bk), dt) ||
        !encode(&tmA, A, K, M, lda * 2, 64, static_cast<uint32_t>(Mp), dt))
        return TG_ERR_LAUNCH;

    SkinnyParams prm;
    const tg_status_t wst = splitk_workspace(dev, stream, pl.grid, max_ctas, &prm);
    if (wst != TG_OK) return wst;
    prm.M = static_cast<int32_t>(M);
    prm.N = static_cast<int32_t>(N);
    prm.K = static_cast<int32_t>(K);
    prm.Mp = static_cast<int32_t>(Mp);
    prm.tiles_n = static_cast<int32_t>(pl.tiles_n);
    prm.k_blocks = static_cast<int32_t>(pl.k_blocks);
    prm.total_units = pl.tiles_n * pl.k_blocks;
    prm.relu = ep.relu;
    prm.e = ep.e;
    prm.out_f32 = ep.out_f32;
    prm.inject = inject;
    prm.timeout_ns = timeout_ns;
    prm.C = C;
    prm.ldc = ldc;

    if (skinny_launch_kernel<T>(tmB, tmA, prm, pl.grid, stream, pl.cluster) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    return TG_OK;
}

using EncodeSwFn = bool (*)(CUtensorMap*, const void*, uint64_t, uint64_t, uint64_t, uint32_t,
                            uint32_t, CUtensorMapDataType, CUtensorMapSwizzle);

// MXFP4 B: Bq (N rows of ceil(K/2) packed bytes along k, stride ldbq) and S
// (ceil(K/32) rows of N scale bytes, stride lds); A fp16.  Pointers 16-byte
// aligned and ldbq, lds multiples of 16, lda of 8 (checked by the caller).
inline tg_status_t skinny_mx_launch(const void* A, const void* Bq, const void* S, void* C,
                                    const tg_plan_t& pl, int64_t M, int64_t N, int64_t K,
                                    int64_t lda, int64_t ldbq, int64_t lds, int64_t ldc,
                                    const EpilogueSpec& ep, cudaStream_t stream, int dev,
                                    int64_t max_ctas, uint64_t timeout_ns, int32_t inject,
                                    EncodeSwFn encode) {
    const int64_t Mp = pl.mma_n;
    CUtensorMap tmBq, tmA, tmS;
    if (!encode(&tmBq, Bq, static_cast<uint64_t>((K + 1) / 2), N, ldbq, 32, 128,
                CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !encode(&tmS, S, N, (K + 31) / 32, lds, 128, kMxBK / 32, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode(&tmA, A, K, M, lda * 2, 64, static_cast<uint32_t>(Mp),
                CU_TENSOR_MAP_DATA_TYPE_FLOAT16, CU_TENSOR_MAP_SWIZZLE_128B))
        return TG_ERR_LAUNCH;
    SkinnyParams prm;
    const tg_status_t wst = splitk_workspace(dev, stream, pl.grid, max_ctas, &prm);
    if (wst != TG_OK) return wst;
    prm.M = static_cast<int32_t>(M);
    prm.N = static_cast<int32_t>(N);
    prm.K = static_cast<int32_t>(K);
    prm.Mp = static_cast<int32_t>(Mp);
    prm.tiles_n = static_cast<int32_t>(pl.tiles_n);
    prm.k_blocks = static_cast<int32_t>(pl.k_blocks);
    prm.total_units = pl.tiles_n * pl.k_blocks;
    prm.relu = ep.relu;
    prm.e = ep.e;
    prm.out_f32 = ep.out_f32;
    prm.inject = inject;
    prm.timeout_ns = timeout_ns;
    prm.C = C;
    prm.ldc = ldc;
    if (skinny_mx_launch_kernel(tmBq, tmA, tmS, prm, pl.grid, stream) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    return TG_OK;
}

}  // namespace tg
