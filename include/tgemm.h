/*
 * libtgemm — dense FP16 GEMM for GB300 (sm_103a), C ABI.
 *
 *   C = epi(A · B)      A: M×K, B: K×N, C: M×N, all fp16, row-major,
 *                       fp32 accumulation, one rounding to fp16 at the end,
 *                       epi = identity or ReLU on the fp32 accumulator.
 *
 * The operation is the tiled GEMM of the TileLang pages:
 *   - "5分钟上手TileLang" (0539edu.com), section "安装与第一个内核": A (M×K)
 *     and B (K×N) fp16, a float32 accumulator fragment, C fp16; the official
 *     quickstart carries a fused ReLU epilogue;
 *   - same page, section "避坑与调参": the accumulator stays float32 and is
 *     written back as fp16 only at the last copy;
 *   - "TileLang：让GPU编程像Python一样简单的高性能计算新范式" (coreui.cn):
 *     the ReLU epilogue takes max(C_local, 0) on the float32 accumulator
 *     before the copy to C;
 *   - "TileLang：比 Triton 低一层的 tile 语言" (anrans.github.io), sections
 *     "第一个 kernel：GEMM" and "它生成了什么": one output tile per block,
 *     TMA loads into a multi-stage shared-memory ring guarded by mbarriers,
 *     warp-specialised producer and consumer.
 *
 * Threading: every entry point is thread-safe.  Calls on the same stream are
 * ordered; calls on different streams may overlap (each stream gets its own
 * split-K workspace).
 */
#ifndef TGEMM_H
#define TGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TG_EPI_NONE = 0, /* C = fp16(acc)              */
    TG_EPI_RELU = 1  /* C = fp16(acc > 0 ? acc : 0) (so -0 and NaN become +0) */
} tg_epilogue_t;

typedef enum {
    TG_OK = 0,
    TG_ERR_INVALID_VALUE = 1,      /* bad size, leading dimension, pointer or epilogue   */
    TG_ERR_MISALIGNED = 2,         /* pointer not 16-byte aligned or ld not a multiple of 8 */
    TG_ERR_UNSUPPORTED_DEVICE = 3, /* no CUDA device, or the current one is not sm_103     */
    TG_ERR_LAUNCH = 4,             /* a CUDA launch or runtime call failed                 */
    TG_ERR_NO_MEMORY = 5,          /* the library could not allocate its workspace         */
    TG_ERR_TIMEOUT = 6             /* a kernel gave up on a wait and returned early        */
} tg_status_t;

/*
 * tg_gemm_f16 — C = epi(A·B), asynchronous on `stream`.
 *
 * A   device pointer, fp16, row-major M×K, row stride lda elements (lda ≥ K).
 * B   device pointer, fp16, row-major K×N, row stride ldb elements (ldb ≥ N).
 * C   device pointer, fp16, row-major M×N, row stride ldc elements (ldc ≥ N).
 *     Only the M×N elements are written; padding columns are left untouched.
 * M, N, K   sizes, each in [0, 2^31 - 1].  M == 0 or N == 0: nothing is done
 *     and TG_OK is returned.  K == 0: C is filled with epi(0) = +0 (A and B
 *     may then be NULL and lda/ldb are ignored).
 * epilogue  TG_EPI_NONE or TG_EPI_RELU.
 * stream    a cudaStream_t (NULL = the legacy default stream) on the current
 *     device.
 *
 * Layout: A, B and C need only be aligned to their 2-byte elements (else
 * TG_ERR_MISALIGNED); any lda ≥ K, ldb ≥ N, ldc ≥ N is accepted.  The kernels
 * read and write through the tensor memory-access unit, which needs 16-byte
 * aligned rows: an operand whose pointer is not 16-byte aligned or whose
 * leading dimension is not a multiple of 8 is first copied into an aligned
 * staging buffer (per device and stream, grown on demand; growth waits for
 * the stream), and a C in such a layout is computed there and copied back.
 * That costs one extra read and write of the staged matrices.  C must not
 * overlap A or B (not checked).
 * Ownership: the caller owns A, B and C; the library keeps no reference past
 * the work it enqueued on `stream`.  The library owns a split-K workspace
 * per (device, stream): two 64 KB fp32 slots and four counter words per SM
 * (about 20 MB on 152 SMs), allocated by the first call on that stream that
 * runs the M <= 128 kernel or the CTA-pair kernel, and kept until process
 * exit.  If it cannot be allocated, an M <= 128 call returns
 * TG_ERR_NO_MEMORY and a pair-kernel call runs without cutting its last
 * wave of tiles into k-pieces (column halves, which need no workspace, are
 * still used).
 * Errors: argument errors are returned before anything is enqueued.  Launch
 * failures return TG_ERR_LAUNCH.  A kernel that gives up on a bounded wait
 * records the fact on the device; tg_sync_status reports it.
 * The current device must be compute capability 10.3 (sm_103).
 * Kernel choice follows tg_plan_f16; the environment variable
 * TGEMM_FORCE_CFG = pair256 | persistent256 | persistent128 | skinny
 * overrides it where the forced kernel applies, and TGEMM_GROUP_M sets the
 * raster group height (both for tests and tile sweeps).
 * CUDA graphs: once a call that runs the M <= 128 kernel or the CTA-pair
 * kernel has run on a stream outside capture (allocating that stream's
 * split-K workspace), calls on that stream can be captured; a graph holding
 * such a call uses the capturing stream's workspace, so it must not run
 * concurrently with other libtgemm work on that stream.
 * Kernels are launched with programmatic dependent launch: each may start its
 * set-up while the previous kernel on the stream finishes, and waits for that
 * kernel's completion before it reads or writes global memory.
 */
tg_status_t tg_gemm_f16(const void* A, const void* B, void* C,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldc,
                        int epilogue, void* stream);

/*
 * tg_gemm_bf16 — the same operation with bfloat16 storage of A, B and C:
 * C = bf16_rne(epi(A·B)), fp32 accumulation.  The pages define the GEMM for
 * fp16 only ("5分钟上手TileLang", section "安装与第一个内核"); bf16 runs on the
 * same tensor-core instruction kind (operand format bf16 instead of f16)
 * through the same kernels, so arguments, layouts, alignment, ownership,
 * errors and kernel choice are exactly those of tg_gemm_f16.
 */
tg_status_t tg_gemm_bf16(const void* A, const void* B, void* C,
                         int64_t M, int64_t N, int64_t K,
                         int64_t lda, int64_t ldb, int64_t ldc,
                         int epilogue, void* stream);

/* ------------------------------------------------------------------------
 * Extended epilogue: bias, residual, fp32 output.
 * ------------------------------------------------------------------------ */

typedef enum {
    TG_DTYPE_F16 = 0,  /* IEEE binary16               */
    TG_DTYPE_BF16 = 1, /* bfloat16                    */
    TG_DTYPE_F32 = 2   /* IEEE binary32 (output only) */
} tg_dtype_t;

typedef struct {
    int32_t activation;   /* tg_epilogue_t: TG_EPI_NONE or TG_EPI_RELU              */
    int32_t out_dtype;    /* tg_dtype_t of C: the input type, or TG_DTYPE_F32       */
    const float* bias;    /* device, N fp32 values (one per column of C), or NULL  */
    const void* residual; /* device, M×N of the input type, row stride ldr, or NULL */
    int64_t ldr;          /* row stride of residual in elements (≥ N when present) */
} tg_epilogue_ex_t;

/*
 * tg_gemm_ex — C = out( act( A·B + bias ) + R ), asynchronous on `stream`:
 *
 *   C[i][j] = out( act( sum_k A[i][k]·B[k][j] + bias[j] ) + R[i][j] )
 *
 * with the sum accumulated in fp32, bias (if given) added to the fp32
 * accumulator, act = identity or ReLU, the residual R (if given, stored in
 * the input type) added after the activation in fp32, and one rounding at
 * the end: round-to-nearest-even to the input type, or none for fp32 output.
 * It widens the element-wise epilogue of the pages — the ReLU taken on the
 * float32 accumulator before the final copy ("TileLang：让GPU编程像Python一样
 * 简单的高性能计算新范式", the T.Parallel loop over C_local; "5分钟上手TileLang",
 * section "安装与第一个内核", whose quickstart carries a fused epilogue) — to
 * the bias, residual and output-type variants a layer's GEMM needs; the pages
 * define none of the three, so their placement (bias before, residual after
 * the activation) is this library's reading.
 *
 * in_dtype  TG_DTYPE_F16 or TG_DTYPE_BF16: the type of A, B and R.
 * A, B, M, N, K, lda, ldb, stream  as for tg_gemm_f16 (any row-major layout;
 *     operands the tensor memory-access unit cannot address are staged).
 * C   device pointer of type epi->out_dtype, row-major M×N, row stride ldc
 *     elements (ldc ≥ N); aligned to its element size.  An fp32 C not
 *     16-byte aligned or with ldc not a multiple of 4 is computed in the
 *     staging buffer and copied back.
 * epi NULL means { TG_EPI_NONE, in_dtype, NULL, NULL, 0 } (plain GEMM).
 *     bias must be 4-byte aligned, residual aligned to its element.  R may be
 *     the same buffer as C (same pointer, ldr == ldc, same 16-bit type): each
 *     element is read before it is overwritten.  Any other overlap of R or
 *     bias with C is undefined.
 * K == 0: C = out(act(bias) + R) (the product is +0).
 * Errors: TG_ERR_INVALID_VALUE for an unknown dtype or activation, an output
 * type that is neither the input type nor fp32, ldr < N, or a NULL C, A or B
 * where needed; TG_ERR_MISALIGNED for a pointer not aligned to its element;
 * otherwise as tg_gemm_f16.
 */
tg_status_t tg_gemm_ex(int32_t in_dtype, const void* A, const void* B, void* C,
                       int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc,
                       const tg_epilogue_ex_t* epi, void* stream);

/* ------------------------------------------------------------------------
 * MXFP4 weights: C = out(act(A · Bdeq + bias) + R), A fp16, B in MXFP4.
 * ------------------------------------------------------------------------ */

/*
 * tg_gemm_mxfp4 — the GEMM with B stored in the OCP Microscaling MXFP4
 * format and dequantised to fp16 inside the library, asynchronous on
 * `stream`:
 *
 *   code(k, n)  4-bit FP4 E2M1 element: byte Bq[n*ldbq + k/2], low nibble for
 *               even k, high nibble for odd k (sign bit, 2 exponent bits with
 *               bias 1, 1 mantissa bit; values 0, ±0.5, ±1, ±1.5, ±2, ±3, ±4, ±6).
 *               B is stored in the [out][in] orientation of a linear layer's
 *               weight: one row of packed codes per column n, k contiguous;
 *   X(k, n)     8-bit E8M0 scale of the block of 32 k holding k:
 *               Bscale[(k/32)*ldbs + n]; its value is 2^(X-127), X = 255 NaN;
 *   Bdeq[k][n]  = fp16_rne(e2m1(code) * 2^(X-127));
 *   C           = out(act(A·Bdeq + bias) + R) exactly as tg_gemm_ex with
 *                 in_dtype TG_DTYPE_F16 (fp32 accumulation, one rounding).
 *
 * The pages name low-bit weight GEMMs as the largest mixed-precision gain
 * ("5分钟上手TileLang", section "H100 实测": WFP4; section "进阶方向":
 * dequantize_gemm with W4A8 and MXFP4; "TileLang：让GPU编程像Python一样
 * 简单的高性能计算新范式": WINT2AFP16) but define no format; MXFP4 as
 * specified by OCP, with fp16 activations, is this library's reading.
 *
 * A        device, fp16, row-major M×K, row stride lda ≥ K, 2-byte aligned
 *          (other layouts than 16-byte aligned rows are staged).
 * Bq       device, N rows of ceil(K/2) bytes, row stride ldbq ≥ ceil(K/2);
 *          Bq 16-byte aligned and ldbq a multiple of 16 (else
 *          TG_ERR_MISALIGNED).  A spare high nibble (odd K) is ignored.
 * Bscale   device, ceil(K/32) rows of N bytes, row stride ldbs ≥ N; 16-byte
 *          aligned, ldbs a multiple of 16 (else TG_ERR_MISALIGNED).
 * C, ldc, epi, stream  as tg_gemm_ex with in_dtype TG_DTYPE_F16 (epi NULL =
 *          plain fp16 output; the residual, if any, is fp16).
 * M ≤ 128: a split-K kernel streams Bq and Bscale once and decodes them
 *          into tensor memory (about 0.53 bytes per weight instead of 2).
 * M > 128: Bq is dequantised once into a per-(device, stream) fp16 buffer of
 *          K × roundup(N, 8) elements (grown on demand; growth waits for the
 *          stream), then the fp16 GEMM runs on it.  TGEMM_FORCE_CFG =
 *          pair256 | persistent256 | persistent128 takes this path for any M.
 * K == 0:  C = out(act(bias) + R); A, Bq and Bscale may be NULL.
 * Errors: as tg_gemm_ex, plus TG_ERR_INVALID_VALUE for ldbq < ceil(K/2) or
 * ldbs < N, and TG_ERR_MISALIGNED for the Bq / Bscale alignment rules above.
 */
tg_status_t tg_gemm_mxfp4(const void* A, const void* Bq, const void* Bscale, void* C,
                          int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldbq, int64_t ldbs, int64_t ldc,
                          const tg_epilogue_ex_t* epi, void* stream);

/* ------------------------------------------------------------------------
 * 2:4 structured-sparse A: C = out(act(A · B + bias) + R).
 * ------------------------------------------------------------------------ */

/*
 * tg_gemm_sp24 — the GEMM with A 2:4 structured-sparse, on the sparse tensor
 * cores (tcgen05.mma.sp), asynchronous on `stream`.  A (M×K) has at most two
 * nonzeros in every aligned group of four k and is passed compressed:
 *
 *   Ac[i][2G + h]  the h-th kept value (h = 0, 1; increasing k) of group G
 *                  (k = 4G .. 4G+3), of type in_dtype, row stride ldac;
 *   E[i][w]        32-bit metadata word w (k = 32w .. 32w+31), row stride lde
 *                  words: group g of the word in bits 4g .. 4g+3, the low two
 *                  bits the position (0..3) of the first kept value, the high
 *                  two the second; first < second in every group.
 *
 * The dense A (kept values at their positions, +0 elsewhere) then enters
 *   C[i][j] = out( act( sum_k A[i][k]·B[k][j] + bias[j] ) + R[i][j] )
 * exactly as in tg_gemm_ex (fp32 accumulation, one rounding).  The pages name
 * the operation — T.gemm_sp on 2:4 sparse tensor cores ("TileLang：让GPU编程像
 * Python一样简单的高性能计算新范式") — without a storage format; this packing of
 * positions is the library's reading (the form the tensor core consumes).
 *
 * in_dtype  TG_DTYPE_F16 or TG_DTYPE_BF16 (Ac, B, R).
 * K         a multiple of 32 (else TG_ERR_INVALID_VALUE).
 * Ac, E, B  device; 16-byte aligned with ldac and ldb multiples of 8 elements
 *           and lde a multiple of 4 words (else TG_ERR_MISALIGNED); ldac ≥
 *           K/2, lde ≥ K/32, ldb ≥ N.
 * C         of epi->out_dtype, 16-byte aligned with 16-byte aligned rows (else
 *           TG_ERR_MISALIGNED); no staging on this entry point.
 * epi       as tg_gemm_ex (NULL: plain output in the input type).
 * Metadata that breaks first < second gives undefined values in its row of
 * C (it is not checked on the device).  K == 0: C = out(act(bias) + R).
 */
tg_status_t tg_gemm_sp24(int32_t in_dtype, const void* Ac, const void* E, const void* B,
                         void* C, int64_t M, int64_t N, int64_t K,
                         int64_t ldac, int64_t lde, int64_t ldb, int64_t ldc,
                         const tg_epilogue_ex_t* epi, void* stream);

/*
 * tg_sync_status — wait for `stream`, then report (and clear) a device-side
 * timeout recorded by any libtgemm kernel on the current device since the
 * last call.  Returns TG_OK, TG_ERR_TIMEOUT, or TG_ERR_LAUNCH if the stream
 * reports a CUDA error.
 */
tg_status_t tg_sync_status(void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* tg_status_string(tg_status_t status);

/* Library version string, e.g. "libtgemm 0.1.0 (sm_103a)". */
const char* tg_version(void);

/* ------------------------------------------------------------------------
 * Host-side planning (pure functions: no CUDA calls, usable without a GPU).
 * ------------------------------------------------------------------------ */

typedef enum {
    TG_KERNEL_NONE = 0,       /* M == 0 or N == 0                                   */
    TG_KERNEL_FILL = 1,       /* K == 0: C = 0                                      */
    TG_KERNEL_PERSISTENT = 2, /* 128×BN tiles, persistent CTAs, TMEM accumulator    */
    TG_KERNEL_SKINNY = 3      /* M ≤ 128: C^T = B^T·A^T tiles with split-K          */
} tg_kernel_t;

typedef struct {
    int32_t kernel;       /* tg_kernel_t                                        */
    int32_t bm, bn, bk;   /* output tile (rows of C, columns of C) and k step   */
    int32_t stages;       /* shared-memory ring depth                           */
    int32_t mma_m, mma_n; /* tensor-core instruction shape                      */
    int64_t tiles_m, tiles_n, k_blocks;
    int64_t num_tiles;
    int64_t grid;         /* CTAs launched                                      */
    int32_t threads;      /* threads per CTA                                    */
    int32_t group_m;      /* raster: tiles_m blocks walked per group            */
    int64_t smem_bytes;   /* dynamic shared memory per CTA                      */
    int64_t ring_bytes;   /* of which the operand ring                          */
    int64_t split_k;      /* k-ranges per output tile (skinny: maximum; CTA   */
                          /* pairs: pieces per tile of the last wave)           */
    int64_t workspace_bytes; /* device scratch used (split-K partial sums)      */
    int32_t cluster;      /* CTAs per cluster: 2 = tcgen05 CTA pair (256-row MMA); */
                          /* M <= 128: 4 = a tile's four k-pieces together     */
    int32_t split_n;      /* CTA pairs: column halves (1 or 2) per tile of the  */
                          /* last wave; 0 for the other kernels                 */
} tg_plan_t;

/*
 * tg_plan_f16 — the launch plan tg_gemm_f16 uses for these sizes on a device
 * with `num_sms` multiprocessors.  Returns TG_ERR_INVALID_VALUE for negative
 * or oversized dimensions or num_sms < 1.
 */
tg_status_t tg_plan_f16(int64_t M, int64_t N, int64_t K, int32_t num_sms, tg_plan_t* plan);

/*
 * tg_plan_f16_limits — the same plan on a device that holds at most
 * `max_pairs` CTA pairs of the pair kernel, and `max_quads_narrow` /
 * `max_quads_wide` clusters of four skinny CTAs (M ≤ 64 / M ≤ 128), at once.
 * Clusters must sit inside one GPC, so these can be below num_sms / 2 and
 * num_sms / 4; tg_plan_f16 assumes they are not.  With the limits of the
 * current device (tg_device_limits) the result is exactly the shape
 * tg_gemm_f16 launches: pairs beyond max_pairs are never launched (none:
 * one-CTA tiles), and a skinny grid whose clusters would not all fit at
 * once launches without clusters.  Returns TG_ERR_INVALID_VALUE for
 * negative limits or as tg_plan_f16.
 */
tg_status_t tg_plan_f16_limits(int64_t M, int64_t N, int64_t K, int32_t num_sms,
                               int32_t max_pairs, int32_t max_quads_narrow,
                               int32_t max_quads_wide, tg_plan_t* plan);

/*
 * tg_device_limits — the limits above for the current device (occupancy
 * queries made once per device; needs a GB300).  Returns
 * TG_ERR_UNSUPPORTED_DEVICE on any other device, TG_ERR_INVALID_VALUE for a
 * NULL output.
 */
tg_status_t tg_device_limits(int32_t* num_sms, int32_t* max_pairs, int32_t* max_quads_narrow,
                             int32_t* max_quads_wide);

/*
 * tg_tile_coord — which (m block, n block) tile number `tile` of a plan maps
 * to; the persistent kernel walks tiles in this order (column-major inside
 * groups of plan->group_m row blocks, so consecutive CTAs share B panels in
 * L2).  Returns TG_ERR_INVALID_VALUE if `tile` is out of range.
 */
tg_status_t tg_tile_coord(const tg_plan_t* plan, int64_t tile, int64_t* m_blk, int64_t* n_blk);

/*
 * tg_ring_bytes — bytes of a shared-memory ring of `stages` stages, each
 * holding one bm×bk tile of A and one bk×bn tile of B of `elem_bytes`-byte
 * elements.  "TileLang：比 Triton 低一层的 tile 语言", section "练习",
 * exercises 1–2 work this out for 128/128/64 fp16: 32 KB per stage, 96 KB
 * for 3 stages.  Returns -1 for non-positive arguments.
 */
int64_t tg_ring_bytes(int32_t bm, int32_t bn, int32_t bk, int32_t stages, int32_t elem_bytes);

/* ------------------------------------------------------------------------
 * Fault-path hooks (for tests of the timeout path; they never fault a GPU).
 * ------------------------------------------------------------------------ */

/* Upper bound, in nanoseconds, on every wait inside libtgemm kernels launched
 * after this call (default 2 000 000 000).  0 restores the default. */
void tg_debug_set_wait_timeout_ns(uint64_t ns);

/* mode 1: the next persistent/skinny launch withholds its first
 * "accumulator ready" signal, so its epilogue waits out the timeout and the
 * kernel returns early with TG_ERR_TIMEOUT recorded.  mode 0: off.  The
 * setting applies to exactly one launch. */
void tg_debug_inject(int32_t mode);

/* The shape of the last tg_gemm_f16 / tg_gemm_bf16 / tg_gemm_ex launch made
 * by the calling thread (tg_gemm_f16_noalloc's too): its plan, with grid,
 * split_k, cluster and split_n as actually launched.  These differ from the
 * plan only if the pair kernel's split-K workspace could not be allocated
 * (the last wave then runs without k-pieces).  Returns TG_ERR_INVALID_VALUE
 * for NULL. */
tg_status_t tg_debug_last_launch(tg_plan_t* plan);

/* Tensor maps served from the library's map cache (hits) and encoded anew
 * (misses) since the library was loaded.  A map depends only on the
 * address, extents, row stride, box and modes it encodes, and the cache is
 * keyed by all of them, so a hit is always the map the call needs. */
void tg_debug_map_cache_stats(uint64_t* hits, uint64_t* misses);

/* ------------------------------------------------------------------------
 * Host buffers in and out.
 * ------------------------------------------------------------------------ */

/*
 * tg_gemm_f16_host — C = epi(A·B) with A, B and C in host memory,
 * asynchronous on `stream`.  The pages' GEMM (the tiled fp16 product with
 * the ReLU epilogue: "TileLang：让GPU编程像Python一样简单的高性能计算新范式",
 * the GEMM example) run end to end: the copies to and from the device are
 * part of the call.
 *
 * A, B, C   HOST pointers, fp16, row-major, with row strides lda ≥ K,
 *     ldb ≥ N, ldc ≥ N elements, 2-byte aligned (else TG_ERR_MISALIGNED).
 *     Page-locked (pinned) memory lets the copies overlap the computation;
 *     pageable memory works but each copy then waits for the host.
 * M, N, K, epilogue, stream   as for tg_gemm_f16.
 *
 * The call uploads A, then walks N in blocks of columns (at most 8: 1024
 * columns, then doubling up to 8192, the last taking the rest): for each
 * block the library copies that
 * block of B up on a copy stream of its own, runs the GEMM of the block on
 * `stream`, and copies that block of C down on a second copy stream, ordered
 * by events, so uploads, products and downloads of different blocks overlap.
 * `stream` waits for the last download: once `stream` completes (e.g.
 * cudaStreamSynchronize), C holds the result.  Work already enqueued on
 * `stream` completes before the call's first copy starts.
 * Ownership: the caller owns A, B and C and must keep them alive and
 * unmodified (C unread) until `stream` completes.  The library owns device
 * copies of A, B and C and the two copy streams, per (device, stream), grown
 * on demand (growth waits for earlier calls on that stream) and kept until
 * process exit.
 * Errors: as tg_gemm_f16; TG_ERR_NO_MEMORY if the device copies cannot be
 * allocated; TG_ERR_LAUNCH if a copy or launch cannot be enqueued.
 */
tg_status_t tg_gemm_f16_host(const void* A, const void* B, void* C,
                             int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, int64_t ldc,
                             int epilogue, void* stream);

/* ------------------------------------------------------------------------
 * Entry point that allocates nothing.
 * ------------------------------------------------------------------------ */

/* Size of the scratch array inside the library that tg_gemm_f16_noalloc uses. */
#define TG_NOALLOC_SCRATCH_BYTES ((int64_t)24 * 1024 * 1024)

/*
 * tg_gemm_f16_noalloc — C = epi(A·B) for 1 ≤ M ≤ 128 without allocating any
 * device memory.  The pages have no counterpart for this entry point: it
 * exists for callers that cannot allocate device memory at call time, e.g. a
 * service that handed all device memory to its own pool allocator at
 * start-up (a late cudaMalloc would fail or fragment that pool), or code in a
 * phase where a cudaMalloc, which may synchronise the whole device, must not
 * stall other streams.
 *
 * It runs the same split-K kernel that tg_gemm_f16 uses for M ≤ 128, with its
 * scratch (fp32 partial sums and piece counters) in a fixed array of
 * TG_NOALLOC_SCRATCH_BYTES (24 MiB) inside the library; every device that
 * loads the library holds that array until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, ownership of A, B and C, and argument errors are those of
 * tg_gemm_f16, except that it has no staging buffer: A, B, C must be 16-byte
 * aligned and lda, ldb, ldc multiples of 8 (else TG_ERR_MISALIGNED).
 * Additionally:
 *   - M > 128 returns TG_ERR_INVALID_VALUE (the split-K kernel covers
 *     M ≤ 128 only); so does a problem whose split needs more scratch than the
 *     array holds (more than 191 CTAs, i.e. a device with more than 191 SMs).
 *   - K == 0 fills C with +0 and uses no scratch; M == 0 or N == 0 is a no-op.
 *   - Set-up: the first call on each device (with that device current) looks
 *     up the array's device address and clears its counter words on `stream`.
 *     Make that first call before any stream capture begins.
 *   - Every call shares the one array, which keeps what the last call left in
 *     it.  Calls whose kernels overlap on the GPU (e.g. on two streams with no
 *     ordering between them) race on it and give wrong results: order them on
 *     one stream or with events.
 */
tg_status_t tg_gemm_f16_noalloc(const void* A, const void* B, void* C,
                                int64_t M, int64_t N, int64_t K,
                                int64_t lda, int64_t ldb, int64_t ldc,
                                int epilogue, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_H */
