// sm_103a device primitives for libtgemm: mbarriers, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM allocation, MMA issue, commit, TMEM loads) and the shared-memory
// matrix / instruction descriptors the tensor core reads.  Hand-written inline PTX.
//
// Every wait in this library is bounded: mbar_wait() gives up after a
// caller-given number of nanoseconds (measured on %globaltimer) or as soon as
// another role of the same CTA has raised the CTA's abort flag.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace tg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ dependent launch
//
// Every GEMM kernel of this library is launched with programmatic stream
// serialisation allowed (the staging copy and the MXFP4 dequantisation are
// plain launches that release their dependents early; the K = 0 fills are
// plain launches): its CTAs may be placed on SMs that the previous
// kernel in the stream has already left, and run their set-up (barrier
// initialisation, tensor-memory allocation, descriptor prefetch) while that
// kernel's last CTAs finish.  grid_dependency_wait() then blocks until the
// previous kernel has completed and its memory writes are visible, so nothing
// before it may touch global memory that another kernel writes.  Where the
// previous work is not a kernel (a copy, an event wait) it is a plain stream
// dependency and the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel in the stream be scheduled onto SMs as they free up.
// It cannot start before this one's CTAs are all placed, and it reads
// nothing this one writes before its own grid_dependency_wait().
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ global atomics

// Returns the old value; orders this thread's earlier writes before the add
// and its later reads after it, at GPU scope.
__device__ __forceinline__ uint32_t atomic_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

inline void set_dependent_launch(cudaLaunchAttribute& a) {
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tensor core).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// The same, suspending the thread until the phase completes or about
// `hint_ns` nanoseconds have passed (the instruction's suspend-time hint).
// A waiting warp then sleeps instead of re-issuing the test: the roles of a
// kernel share their SM's schedulers, and waiting warps that kept polling
// took issue slots from the working ones.
__device__ __forceinline__ uint32_t mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                        uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok;
}

// Longest single suspension of a waiting thread; the give-up limit and the
// abort flag are checked between suspensions.
constexpr uint32_t kWaitSleepNs = 200000;

__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                            const volatile int* abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// Wait until the phase of `bar` with parity `parity` has completed.  Returns
// false if it did not within `timeout_ns`, or if *abort_flag became non-zero.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, timeout_ns, abort_flag);
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* desc) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled as
// transaction bytes on `bar`.  x is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* desc, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Same, with an L2 eviction-priority hint (a createpolicy value).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* desc, uint32_t bar,
                                                 int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Plain bulk copy global → this CTA's shared memory, completing `bytes`
// transaction bytes on `bar` (addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// L2 prefetch of one box of a 2-D tensor map.  A prefetch only fills L2,
// which every SM and TMA unit reads through, so it may be issued before
// grid_dependency_wait(): the loads after the wait still see the previous
// kernel's writes.
__device__ __forceinline__ void tma_prefetch_2d(const void* desc, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(desc),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled store of one box from shared memory (clipped at the tensor edges).
__device__ __forceinline__ void tma_store_2d(const void* desc, uint32_t src, int32_t x,
                                             int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(desc)),
        "r"(x), "r"(y), "r"(src)
        : "memory");
}

// Same, with an L2 eviction-priority hint for the written lines.
__device__ __forceinline__ void tma_store_2d_hint(const void* desc, uint32_t src, int32_t x,
                                                  int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint"
        " [%0, {%1, %2}], [%3], %4;" ::"l"(reinterpret_cast<uint64_t>(desc)),
        "r"(x), "r"(y), "r"(src), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed bulk groups are still in flight at all.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order generic-proxy global-memory accesses before later async-proxy (bulk
// copy) accesses of global memory.  Writers of data that another thread will
// bulk-copy issue it after their stores; the reader issues it after the
// acquire that observed those writes and before its bulk copies.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// ------------------------------------------------------------------ tcgen05

// One full warp: allocate `ncols` TMEM columns (power of two ≥ 32); the base
// address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] · B[smem]^T, fp16 inputs, fp32 accumulator, one CTA.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-collective forms: every lane of a converged warp executes the call
// with the same operands and one elected lane issues the instruction.  The
// issuing loop then runs warp-uniform, so its descriptors and addresses stay
// warp-uniform values.  Measured on GB300 with one CTA issuing 8192 MMAs of
// 128×64×16, A in tensor memory: 32 cycles per MMA (the tensor pipe's rate)
// against 45.5 issued from a single-lane branch.
__device__ __forceinline__ void mma_f16_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// A operand in tensor memory (K-major: lane = row, 32-bit column = two
// consecutive k, lower k in the low half), B in shared memory.
__device__ __forceinline__ void mma_f16_ts_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(bar)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Warp-collective: thread t of the warp reads TMEM lane (lane base + t),
// columns [col, col + 32) of `taddr`; waits for completion before returning.
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// The same for columns [col, col + 64): one load, one wait.
__device__ __forceinline__ void tmem_ld_x64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}

// ------------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
//   K-major operand (rows of 64 fp16 along K, 8-row swizzle atoms of 1 KB):
//     lbo unused (16), sbo = byte distance between 8-row groups.
//   MN-major operand (rows of 64 fp16 along M/N, one row per k):
//     lbo = byte distance between 64-element M/N chunks,
//     sbo = byte distance between groups of 8 k-rows.
// The tile base must be 1024-byte aligned; advancing the start address inside
// a swizzle atom selects a later k slice.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
           (1ull << 46) |  // descriptor version for tcgen05
           (2ull << 61);   // swizzle mode: 128 B
}

// Instruction descriptor for tcgen05.mma kind::f16 with 16-bit A and B of
// format `ab_fmt` (0 = f16, 1 = bf16; A and B always share it) and an fp32
// accumulator.  a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n, bool a_mn, bool b_mn,
                                                     uint32_t ab_fmt = 0) {
    return (1u << 4)                                  // D format: f32
           | (ab_fmt << 7) | (ab_fmt << 10)           // A, B format
           | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16)
           | (static_cast<uint32_t>(n >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);   // M / 16
}

// The two 16-bit element types: operand format code for the instruction
// descriptor, and the epilogue's fp32 → storage rounding (nearest, ties to
// even), two values packed per 32-bit word (first in the low half).
template <typename T>
struct Elem16;

template <>
struct Elem16<__half> {
    static constexpr uint32_t kFmt = 0;
    __device__ static __forceinline__ uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static __forceinline__ __half from_float(float x) { return __float2half_rn(x); }
    __device__ static __forceinline__ float to_float(__half x) { return __half2float(x); }
};

template <>
struct Elem16<__nv_bfloat16> {
    static constexpr uint32_t kFmt = 1;
    __device__ static __forceinline__ uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static __forceinline__ __nv_bfloat16 from_float(float x) {
        return __float2bfloat16_rn(x);
    }
    __device__ static __forceinline__ float to_float(__nv_bfloat16 x) {
        return __bfloat162float(x);
    }
};

// ------------------------------------------------------------------ CTA pairs (cta_group::2)
//
// A cluster of two CTAs on two SMs shares one 256-row MMA: each CTA holds
// half of A (its 128 rows) and half of B (half the N columns) in its own
// shared memory at the same offsets; the even CTA issues the MMA, whose
// result rows 0-127 land in its TMEM and rows 128-255 in the peer's.

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address, in the cluster shared window, of the variable at shared::cta
// address `addr` in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive (release, cluster scope) on an mbarrier given by its cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// TMA load into this CTA's shared memory whose completion bytes are counted
// on an mbarrier that may live in the peer CTA (cluster address `bar`).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* desc, uint32_t bar,
                                                 int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The same with an L2 eviction-priority hint (a createpolicy value).
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const void* desc, uint32_t bar,
                                                      int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem of both CTAs] (+)= A · B^T over the CTA pair; issued by the even CTA.
__device__ __forceinline__ void mma_f16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One 64-k stage of a one-CTA kernel: four MMAs, A and B descriptors advanced
// by A_STEP and B_STEP (16-byte units) per 16 k, and the stage's release
// commit, issued by one elected lane of a converged warp in one block.
// first != 0: the first MMA overwrites D.
template <uint32_t A_STEP, uint32_t B_STEP>
__device__ __forceinline__ void stage4_mma_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                    uint64_t b_desc, uint32_t idesc,
                                                    uint32_t first, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b64 a, b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.eq.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "add.u64 a, %1, %6;\n\tadd.u64 b, %2, %7;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
        "add.u64 a, a, %6;\n\tadd.u64 b, b, %7;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
        "add.u64 a, a, %6;\n\tadd.u64 b, b, %7;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
        "}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(first), "r"(bar), "n"(A_STEP), "n"(B_STEP)
        : "memory");
}

// One 128-k stage of the dense pair kernel: eight MMAs of 256 × 256 × 16
// over the pair and the stage's release commit (multicast to both CTAs),
// issued by one elected lane of a converged warp in one block.  MMA k reads
// A at a_desc + 1024 (k / 4) + 2 (k % 4) (64-k boxes of 16 KB, 32 B per 16 k)
// and B at b_desc + 128 k (16 k rows of 2 KB), in descriptor address units of
// 16 bytes.  first != 0: the first MMA overwrites D.
__device__ __forceinline__ void pair_stage_mma_elect(uint32_t d_tmem, uint64_t a_desc,
                                                     uint64_t b_desc, uint32_t idesc,
                                                     uint32_t first, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b64 a, b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.eq.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "add.u64 a, %1, 2;\n\tadd.u64 b, %2, 128;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, t;\n\t"
        "add.u64 a, %1, 4;\n\tadd.u64 b, %2, 256;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, t;\n\t"
        "add.u64 a, %1, 6;\n\tadd.u64 b, %2, 384;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, t;\n\t"
        "add.u64 a, %1, 1024;\n\tadd.u64 b, %2, 512;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, t;\n\t"
        "add.u64 a, %1, 1026;\n\tadd.u64 b, %2, 640;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, t;\n\t"
        "add.u64 a, %1, 1028;\n\tadd.u64 b, %2, 768;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, t;\n\t"
        "add.u64 a, %1, 1030;\n\tadd.u64 b, %2, 896;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, t;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%5], %6;\n\t"
        "}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(first), "r"(bar),
        "h"(static_cast<uint16_t>(0x3))
        : "memory");
}

// Arrive once on the mbarrier at shared::cta offset `bar` in every CTA of
// `cta_mask` when this thread's earlier tcgen05 operations have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// ------------------------------------------------------------------ misc

__device__ __forceinline__ float relu_f32(float x) { return x > 0.0f ? x : 0.0f; }

}  // namespace tg
