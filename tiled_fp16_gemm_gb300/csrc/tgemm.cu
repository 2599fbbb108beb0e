// libtgemm host side: argument validation, launch planning, tensor-map
// encoding and kernel launch for C = epi(A·B) (fp16 in, fp32 accumulate,
// fp16 out) on sm_103a.  The C ABI is declared in include/tgemm.h.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <map>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tgemm.h"
#include "copy_matrix.cuh"
#include "gemm_persistent.cuh"
#include "gemm_pair.cuh"
#include "gemm_sparse_pair.cuh"
#include "gemm_skinny.cuh"
#include "gemm_sparse.cuh"
#include "sparse_plan.h"
#include "tile_schedule.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = 2147483647LL;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int32_t> g_inject{0};

void noalloc_reset_counters(int dev);  // defined with the no-allocation entry point below

// ------------------------------------------------------------------ planning

constexpr int kBigBN = 256, kBigStages = 4;
constexpr int kMidBN = 128, kMidStages = 6;
// 128×64 tiles for problems whose 128×128 tiles would fill at most half the
// SMs: twice the CTAs, each loading 24 KB per 64-deep stage instead of 32 KB.
constexpr int kSmallBN = 64, kSmallStages = 8;
constexpr int kGroupM = 16;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

void plan_persistent(int64_t M, int64_t N, int64_t K, int32_t num_sms, int bn, int stages,
                     int64_t smem, tg_plan_t* p) {
    p->kernel = TG_KERNEL_PERSISTENT;
    p->bm = 128;
    p->bn = bn;
    p->bk = 64;
    p->stages = stages;
    p->mma_m = 128;
    p->mma_n = bn;
    p->tiles_m = ceil_div(M, 128);
    p->tiles_n = ceil_div(N, bn);
    p->k_blocks = ceil_div(K, 64);
    p->num_tiles = p->tiles_m * p->tiles_n;
    p->grid = p->num_tiles < num_sms ? p->num_tiles : num_sms;
    p->threads = 192;
    p->group_m = static_cast<int32_t>(p->tiles_m < kGroupM ? p->tiles_m : kGroupM);
    p->smem_bytes = smem;
    p->ring_bytes = tg_ring_bytes(128, bn, 64, stages, 2);
    p->split_k = 1;
    p->workspace_bytes = 0;
    p->cluster = 1;
}

// Pair kernel ring: 3 stages of 128 k (64 KB per CTA each).  The MMA thread
// waits and commits once per stage, so 8 MMAs per stage instead of 4 leave it
// more of each stage's 1024 tensor cycles; measured on the 8192×28672×4096
// workload against 6 stages of 64 k: 1.144 ms vs 1.171 ms, same result bits.
constexpr int kPairStages = 3;
constexpr int kPairBK = 128;  // k per ring stage of the pair kernel
using PairCfgT = tg::PairCfg<kPairStages, kPairBK>;
// 16 blocks of 256 rows = 4096 rows per raster group: a wave of 76 pair tiles
// then spans 16 × ~5 tiles (A 32 MB + B 10 MB in L2) and B is reread M/4096
// times.  Swept on the 8192×28672×4096 workload: 2: 1450, 4: 1528, 8: 1589,
// 16: 1629, 32: 1552 TFLOP/s.
constexpr int kPairGroupM = 16;

// 2:4 sparse pair kernel: 48 KB of operands per stage and CTA.  The plain
// build runs 4 stages with one staging buffer per epilogue warp; the full
// build (bias, residual, fp32 C) keeps two buffers, which leaves room for 3.
constexpr int kSpPairStages = 3;
constexpr int kSpPairStagesPlain = 4;

// What bounds a launch on one device: its SMs, the CTA pairs of the pair
// kernel that fit on it at once, and the clusters of four skinny CTAs (Mp <=
// 64, Mp <= 128) that do.  Clusters must sit inside one GPC, so the last
// two can be below num_sms / 2 and num_sms / 4.
struct PlanLimits {
    int32_t num_sms;
    int32_t pairs;
    int32_t quads[2];
};

tg_status_t plan_limited(int64_t M, int64_t N, int64_t K, const PlanLimits& lim,
                         tg_plan_t* plan);

PlanLimits nominal_limits(int32_t num_sms) {
    PlanLimits l;
    l.num_sms = num_sms;
    l.pairs = num_sms / 2;
    l.quads[0] = l.quads[1] = num_sms / 4;
    return l;
}

// 256×256 tiles on at most `pairs` CTA pairs (two CTAs per pair).
void plan_pair(int64_t M, int64_t N, int64_t K, int32_t pairs, tg_plan_t* p) {
    p->kernel = TG_KERNEL_PERSISTENT;
    p->bm = 256;
    p->bn = 256;
    p->bk = kPairBK;
    p->stages = kPairStages;
    p->mma_m = 256;
    p->mma_n = 256;
    p->tiles_m = ceil_div(M, 256);
    p->tiles_n = ceil_div(N, 256);
    p->k_blocks = ceil_div(K, kPairBK);
    p->num_tiles = p->tiles_m * p->tiles_n;
    if (pairs < 1) pairs = 1;
    int32_t P = 1, S = 1, H = 1;
    tg::pair_launch_shape(static_cast<int32_t>(p->num_tiles), pairs,
                          static_cast<int32_t>(p->k_blocks), &P, &S, &H);
    p->grid = 2 * int64_t{P};
    p->threads = 192;
    p->group_m = static_cast<int32_t>(p->tiles_m < kPairGroupM ? p->tiles_m : kPairGroupM);
    p->smem_bytes = PairCfgT::kSmemBytes;
    p->ring_bytes = 2 * tg_ring_bytes(128, 128, kPairBK, kPairStages, 2);  // both CTAs
    // k-pieces or column halves per tile of the last wave, and the partial
    // slots and counters k-pieces use (tile_schedule.h)
    p->split_k = S;
    p->split_n = H;
    p->workspace_bytes = S > 1 ? int64_t{P} * tg::kPairSlotFloats * 4 + 8 * int64_t{P} * 4 : 0;
    p->cluster = 2;
}

// ------------------------------------------------------------------ device state

struct DeviceState {
    bool probed = false;
    bool supported = false;
    int num_sms = 0;
    bool attrs_set = false;
    int max_pairs = 0;  // CTA pairs of the pair kernel that fit on the device at once
    int max_sp_pairs = 0;  // the same for the 2:4 sparse pair kernel
    // clusters of four CTAs of the skinny kernel (Mp <= 64, Mp <= 128) that
    // fit at once; the planner's clusters of a tile's four k-pieces are used
    // only when all of them do
    int max_skinny_quads[2] = {0, 0};
};

std::mutex g_dev_mutex;
DeviceState g_dev[kMaxDevices];

PlanLimits device_limits(const DeviceState& ds) {
    PlanLimits l;
    l.num_sms = ds.num_sms;
    l.pairs = ds.num_sms / 2 < ds.max_pairs ? ds.num_sms / 2 : ds.max_pairs;
    l.quads[0] = ds.max_skinny_quads[0];
    l.quads[1] = ds.max_skinny_quads[1];
    return l;
}

// The shape of the last dense GEMM launch made by the calling thread
// (tg_debug_last_launch): the plan it ran with, and the grid, pieces per
// tile and cluster size it was actually launched with.
thread_local tg_plan_t g_last_launch;

void record_launch(const tg_plan_t& pl, int64_t grid, int64_t split, int32_t cluster,
                   int32_t split_n = -1) {
    g_last_launch = pl;
    g_last_launch.grid = grid;
    g_last_launch.split_k = split;
    g_last_launch.cluster = cluster;
    if (split_n >= 0) g_last_launch.split_n = split_n;  // else as planned
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// Opt every kernel instantiation of element type T into its shared memory.
template <typename T>
cudaError_t set_kernel_attributes() {
    cudaError_t e = cudaFuncSetAttribute(tg::tg_gemm_f16_persistent<kBigBN, kBigStages, T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tg::PersistentCfg<kBigBN, kBigStages>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_f16_persistent<kMidBN, kMidStages, T>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tg::PersistentCfg<kMidBN, kMidStages>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_f16_persistent<kSmallBN, kSmallStages, T>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tg::PersistentCfg<kSmallBN, kSmallStages>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_f16_persistent<kSmallBN, kSmallStages, T, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tg::PersistentCfg<kSmallBN, kSmallStages>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_f16_persistent<kMidBN, kMidStages, T, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tg::PersistentCfg<kMidBN, kMidStages>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_f16_pair<kPairStages, T, kPairBK>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairCfgT::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_f16_pair<kPairStages, T, kPairBK, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairCfgT::kSmemBytes);
    if (e == cudaSuccess) e = tg::skinny_set_attributes<T>();
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_sp24<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tg::SparseCfg::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_sp24<T, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tg::SparseCfg::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_sp24_pair<kSpPairStages, T>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tg::SparsePairCfg<kSpPairStages>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tg::tg_gemm_sp24_pair<kSpPairStagesPlain, T, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tg::SparsePairCfg<kSpPairStagesPlain>::kSmemBytes);
    return e;
}

// How many clusters of `size` CTAs of `kernel` can be resident together
// (clusters must sit inside one GPC, so this can be below num_sms / size);
// 0 if the query fails.
template <typename Kernel>
int max_active_clusters(Kernel kernel, int threads, uint32_t smem, int num_sms, int size) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(size);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(size * (num_sms / size)));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        clusters = 0;
    }
    return clusters;
}

// Returns TG_OK and fills *dev / *st for the current device, or an error.
tg_status_t current_device(int* dev, DeviceState** st) {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
        cudaGetLastError();
        return TG_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    DeviceState& s = g_dev[d];
    if (!s.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) {
            cudaGetLastError();
            return TG_ERR_UNSUPPORTED_DEVICE;
        }
        s.probed = true;
        s.supported = (major == 10 && minor == 3);
        s.num_sms = sms;
    }
    if (!s.supported) return TG_ERR_UNSUPPORTED_DEVICE;
    if (!s.attrs_set) {
        if (set_kernel_attributes<__half>() != cudaSuccess ||
            set_kernel_attributes<__nv_bfloat16>() != cudaSuccess ||
            tg::skinny_mx_set_attributes() != cudaSuccess) {
            cudaGetLastError();
            return TG_ERR_LAUNCH;
        }
        s.max_pairs = max_active_clusters(tg::tg_gemm_f16_pair<kPairStages, __half, kPairBK>,
                                          PairCfgT::kThreads, PairCfgT::kSmemBytes, s.num_sms, 2);
        s.max_sp_pairs = max_active_clusters(tg::tg_gemm_sp24_pair<kSpPairStages, __half>,
                                             tg::SparsePairCfg<kSpPairStages>::kThreads,
                                             tg::SparsePairCfg<kSpPairStages>::kSmemBytes,
                                             s.num_sms, 2);
        const int plain_sp_pairs = max_active_clusters(
            tg::tg_gemm_sp24_pair<kSpPairStagesPlain, __half, false>,
            tg::SparsePairCfg<kSpPairStagesPlain>::kThreads,
            tg::SparsePairCfg<kSpPairStagesPlain>::kSmemBytes, s.num_sms, 2);
        if (plain_sp_pairs < s.max_sp_pairs) s.max_sp_pairs = plain_sp_pairs;
        using NarrowCfg = tg::SkinnyNarrow;
        using WideCfg = tg::SkinnyWide;
        s.max_skinny_quads[0] = max_active_clusters(
            tg::tg_gemm_f16_skinny<NarrowCfg::kStages, 64, __half, NarrowCfg::kBK>,
            tg::skinny_threads(NarrowCfg::kStages, 64, false), NarrowCfg::kSmemBytes, s.num_sms,
            4);
        s.max_skinny_quads[1] = max_active_clusters(
            tg::tg_gemm_f16_skinny<WideCfg::kStages, 128, __half, WideCfg::kBK>,
            tg::skinny_threads(WideCfg::kStages, 128, false), WideCfg::kSmemBytes, s.num_sms, 4);
        s.attrs_set = true;
    }
    *dev = d;
    *st = &s;
    return TG_OK;
}

template <typename T>
constexpr CUtensorMapDataType tensor_map_type() {
    return tg::Elem16<T>::kFmt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// Encoded tensor maps, keyed by everything the encoding depends on.  A map
// holds only the address, extents, stride, box and modes it was made from
// (no device or allocation state), so an entry stays valid for any later
// call with the same key, whatever happened to the memory in between.  A
// repeated call (same pointers, shape and leading dimensions) then skips the
// encoding of its maps.  The table is direct-mapped: a colliding key
// replaces the entry, so its size is fixed.
struct MapKey {
    const void* ptr;
    uint64_t inner, outer, row_bytes;
    uint32_t box_inner, box_outer;
    int32_t dtype, swizzle;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && inner == o.inner && outer == o.outer &&
               row_bytes == o.row_bytes && box_inner == o.box_inner &&
               box_outer == o.box_outer && dtype == o.dtype && swizzle == o.swizzle;
    }
};

struct MapEntry {
    bool used = false;
    MapKey key{};
    CUtensorMap map{};
};

constexpr int kMapCacheSlots = 1024;
std::mutex g_map_mutex;
MapEntry g_map_cache[kMapCacheSlots];
std::atomic<uint64_t> g_map_hits{0}, g_map_misses{0};

uint32_t map_slot(const MapKey& k) {
    uint64_t h = reinterpret_cast<uintptr_t>(k.ptr) * 0x9E3779B97F4A7C15ull;
    const uint64_t f[] = {k.inner, k.outer, k.row_bytes,
                          (uint64_t{k.box_inner} << 32) | k.box_outer,
                          (static_cast<uint64_t>(static_cast<uint32_t>(k.dtype)) << 32) |
                              static_cast<uint32_t>(k.swizzle)};
    for (uint64_t v : f) h = (h ^ v) * 0x100000001B3ull + (h >> 29);
    return static_cast<uint32_t>((h ^ (h >> 32)) % kMapCacheSlots);
}

// 2-D tensor map: inner (contiguous) extent, outer extent, row stride in
// bytes, box, swizzle, zero fill outside the tensor.  Served from the cache
// above when the same map was made before.
bool encode_2d_sw(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle) {
    MapKey key;
    std::memset(&key, 0, sizeof(key));  // padding too: keys are compared field by field
    key.ptr = ptr;
    key.inner = inner;
    key.outer = outer;
    key.row_bytes = row_bytes;
    key.box_inner = box_inner;
    key.box_outer = box_outer;
    key.dtype = static_cast<int32_t>(dtype);
    key.swizzle = static_cast<int32_t>(swizzle);
    const uint32_t slot = map_slot(key);
    {
        std::lock_guard<std::mutex> lk(g_map_mutex);
        const MapEntry& e = g_map_cache[slot];
        if (e.used && e.key == key) {
            *map = e.map;
            g_map_hits.fetch_add(1, std::memory_order_relaxed);
            return true;
        }
    }
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    g_map_misses.fetch_add(1, std::memory_order_relaxed);
    std::lock_guard<std::mutex> lk(g_map_mutex);
    MapEntry& e = g_map_cache[slot];
    e.used = true;
    e.key = key;
    e.map = *map;
    return true;
}

// The same with the 128-byte swizzle of every 16-bit operand tile.
bool encode_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapDataType dtype) {
    return encode_2d_sw(map, ptr, inner, outer, row_bytes, box_inner, box_outer, dtype,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

// A, B and C maps of the pair / one-CTA kernels.  A: 64 k × 128 rows per box;
// B: 64 columns × b_box_k k rows per box (the kernel's k per stage); C: 32
// rows × 128 bytes per box (64 16-bit or 32 fp32 elements).
template <typename T>
bool encode_abc(CUtensorMap* tmA, CUtensorMap* tmB, CUtensorMap* tmC, const void* A,
                const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                int64_t ldc, bool out_f32, uint32_t b_box_k = 64) {
    constexpr CUtensorMapDataType dt = tensor_map_type<T>();
    return encode_2d(tmA, A, K, M, lda * 2, 64, 128, dt) &&
           encode_2d(tmB, B, N, K, ldb * 2, 64, b_box_k, dt) &&
           (out_f32 ? encode_2d(tmC, C, N, M, ldc * 4, 32, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32)
                    : encode_2d(tmC, C, N, M, ldc * 2, 64, 32, dt));
}

tg::PersistentParams persistent_params(const tg_plan_t& pl, int64_t M, int64_t N, int64_t K,
                                       const tg::EpilogueSpec& ep) {
    tg::PersistentParams prm;
    prm.M = static_cast<int32_t>(M);
    prm.N = static_cast<int32_t>(N);
    prm.K = static_cast<int32_t>(K);
    prm.tiles_m = static_cast<int32_t>(pl.tiles_m);
    prm.tiles_n = static_cast<int32_t>(pl.tiles_n);
    prm.num_tiles = static_cast<int32_t>(pl.num_tiles);
    prm.k_blocks = static_cast<int32_t>(pl.k_blocks);
    prm.group_m = pl.group_m;
    prm.relu = ep.relu;
    prm.inject = g_inject.exchange(0);
    prm.timeout_ns = g_timeout_ns.load();
    prm.e = ep.e;
    prm.out_f32 = ep.out_f32;
    return prm;
}

template <int BN, int STAGES, typename T>
tg_status_t launch_persistent(const void* A, const void* B, void* C, const tg_plan_t& pl,
                              int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                              int64_t ldc, const tg::EpilogueSpec& ep, cudaStream_t stream) {
    CUtensorMap tmA, tmB, tmC;
    if (!encode_abc<T>(&tmA, &tmB, &tmC, A, B, C, M, N, K, lda, ldb, ldc, ep.out_f32 != 0))
        return TG_ERR_LAUNCH;
    const tg::PersistentParams prm = persistent_params(pl, M, N, K, ep);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
    cfg.blockDim = dim3(tg::PersistentCfg<BN, STAGES>::kThreads);
    cfg.dynamicSmemBytes = tg::PersistentCfg<BN, STAGES>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    tg::set_dependent_launch(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    record_launch(pl, pl.grid, 1, 1);
    // the plain epilogue: the variant with the others compiled out (BN <= 128)
    const bool plain = ep.e.bias == nullptr && ep.e.resid == nullptr && ep.out_f32 == 0;
    cudaError_t e = cudaErrorInvalidValue;
    bool launched = false;
    if constexpr (BN <= kMidBN) {
        if (plain) {
            e = cudaLaunchKernelEx(&cfg, tg::tg_gemm_f16_persistent<BN, STAGES, T, false>, tmA,
                                   tmB, tmC, prm);
            launched = true;
        }
    }
    if (!launched)
        e = cudaLaunchKernelEx(&cfg, tg::tg_gemm_f16_persistent<BN, STAGES, T, true>, tmA, tmB,
                               tmC, prm);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    return TG_OK;
}

// The pair kernel: clusters of two CTAs, at most as many pairs as the device
// holds at once (the launch is persistent, so no pair waits for another).
// The last, partial wave of tiles is shared out to otherwise idle pairs as
// column halves or k-pieces (tile_schedule.h).  k-pieces keep their partial
// sums in the stream's split-K workspace, which is set up on the first pair
// launch on the stream whether or not that launch uses it, so a later launch
// inside a graph capture finds it.  Without a workspace only column halves
// are used.
template <typename T>
tg_status_t launch_pair(const void* A, const void* B, void* C, const tg_plan_t& pl, int64_t M,
                        int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        const tg::EpilogueSpec& ep, cudaStream_t stream, int dev,
                        const DeviceState* ds) {
    CUtensorMap tmA, tmB, tmC;
    if (!encode_abc<T>(&tmA, &tmB, &tmC, A, B, C, M, N, K, lda, ldb, ldc, ep.out_f32 != 0,
                       kPairBK))
        return TG_ERR_LAUNCH;
    tg::PersistentParams prm = persistent_params(pl, M, N, K, ep);
    // the planner's shape: P pairs (within the pairs the device holds at
    // once), tail tiles in S k-pieces or H column halves
    int32_t P = static_cast<int32_t>(pl.grid / 2), S = static_cast<int32_t>(pl.split_k),
            H = static_cast<int32_t>(pl.split_n);
    tg::SkinnyParams wsp;
    if (tg::splitk_workspace(dev, stream, ds->num_sms, ds->num_sms, &wsp) == TG_OK &&
        int64_t{P} * tg::kPairSlotFloats <= 2 * int64_t{ds->num_sms} * tg::kSkSlotFloats &&
        8 * P <= 4 * ds->num_sms) {
        prm.ws = wsp.ws;
        prm.counters = wsp.counters;
    } else if (S > 1) {
        // no workspace (out of memory): the same pairs, no k-pieces (column
        // halves need none)
        tg::pair_launch_shape(prm.num_tiles, P, 0, &P, &S, &H);
    }
    prm.split = S;
    prm.split_n = H;
    record_launch(pl, 2 * int64_t{P}, S, 2, H);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    tg::set_dependent_launch(attr[1]);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(2 * P));
    cfg.blockDim = dim3(PairCfgT::kThreads);
    cfg.dynamicSmemBytes = PairCfgT::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e =
        (ep.e.bias == nullptr && ep.e.resid == nullptr && ep.out_f32 == 0)
            ? cudaLaunchKernelEx(&cfg, tg::tg_gemm_f16_pair<kPairStages, T, kPairBK, false>, tmA,
                                 tmB, tmC, prm)
            : cudaLaunchKernelEx(&cfg, tg::tg_gemm_f16_pair<kPairStages, T, kPairBK, true>, tmA,
                                 tmB, tmC, prm);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    return TG_OK;
}

// TGEMM_FORCE_CFG = pair256 | persistent256 | persistent128 | persistent64 | skinny
// overrides the planner's kernel choice (used by tests and tile sweeps);
// ignored where the forced kernel does not apply (skinny needs M <= 128;
// K == 0 always fills).
void apply_forced_config(int64_t M, int64_t N, int64_t K, const PlanLimits& lim,
                         tg_plan_t* pl) {
    if (pl->kernel == TG_KERNEL_NONE || pl->kernel == TG_KERNEL_FILL) return;
    const int32_t num_sms = lim.num_sms;
    const char* f = std::getenv("TGEMM_FORCE_CFG");
    if (f != nullptr && std::strcmp(f, "pair256") == 0 && lim.pairs >= 1)
        plan_pair(M, N, K, lim.pairs, pl);
    else if (f != nullptr && std::strcmp(f, "pair256") == 0)  // no pair fits: one-CTA tiles
        plan_persistent(M, N, K, num_sms, kBigBN, kBigStages,
                        tg::PersistentCfg<kBigBN, kBigStages>::kSmemBytes, pl);
    else if (f != nullptr && std::strcmp(f, "persistent256") == 0)
        plan_persistent(M, N, K, num_sms, kBigBN, kBigStages,
                        tg::PersistentCfg<kBigBN, kBigStages>::kSmemBytes, pl);
    else if (f != nullptr && std::strcmp(f, "persistent128") == 0)
        plan_persistent(M, N, K, num_sms, kMidBN, kMidStages,
                        tg::PersistentCfg<kMidBN, kMidStages>::kSmemBytes, pl);
    else if (f != nullptr && std::strcmp(f, "persistent64") == 0)
        plan_persistent(M, N, K, num_sms, kSmallBN, kSmallStages,
                        tg::PersistentCfg<kSmallBN, kSmallStages>::kSmemBytes, pl);
    else if (f != nullptr && std::strcmp(f, "skinny") == 0 && tg::skinny_applies(M, N, K)) {
        tg::skinny_plan(M, N, K, num_sms, pl);
        if (pl->cluster == 4 && pl->grid / 4 > lim.quads[pl->mma_n > 64 ? 1 : 0]) pl->cluster = 1;
    }
    // TGEMM_GROUP_M = row blocks per raster group of the persistent kernels
    // (for sweeps), clamped to [1, tiles_m].
    const char* g = std::getenv("TGEMM_GROUP_M");
    if (g != nullptr && *g != 0 && pl->kernel == TG_KERNEL_PERSISTENT) {
        long v = std::strtol(g, nullptr, 10);
        if (v < 1) v = 1;
        if (v > pl->tiles_m) v = static_cast<long>(pl->tiles_m);
        pl->group_m = static_cast<int32_t>(v);
    }
}

// Argument checks shared by every entry point: sizes, null pointers, leading
// dimensions, element (2-byte) alignment.  With `tma_layout` also the layout
// the tensor memory-access unit addresses directly: 16-byte aligned pointers
// and leading dimensions that are multiples of 8 elements.
tg_status_t validate(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc, int epilogue, bool tma_layout = true) {
    if (epilogue != TG_EPI_NONE && epilogue != TG_EPI_RELU) return TG_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return TG_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return TG_OK;
    if (C == nullptr || ldc < N) return TG_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || B == nullptr || lda < K || ldb < N)) return TG_ERR_INVALID_VALUE;
    const unsigned mask = tma_layout ? 15u : 1u;
    if ((reinterpret_cast<uintptr_t>(C) & mask) != 0) return TG_ERR_MISALIGNED;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(A) & mask) != 0 ||
                  (reinterpret_cast<uintptr_t>(B) & mask) != 0))
        return TG_ERR_MISALIGNED;
    if (tma_layout && ((ldc & 7) != 0 || (K > 0 && ((lda & 7) != 0 || (ldb & 7) != 0))))
        return TG_ERR_MISALIGNED;
    return TG_OK;
}

bool tma_layout_ok(const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (ld & 7) == 0;
}

int64_t round_up8(int64_t x) { return (x + 7) / 8 * 8; }

// Per-(device, stream) staging buffer for operands in layouts the tensor
// memory-access unit cannot address; grown on demand (growth waits for the
// stream, so it cannot happen inside a stream capture).
struct Staging {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_staging_mutex;
std::map<std::pair<int, cudaStream_t>, Staging> g_staging;

tg_status_t staging_buffer(int dev, cudaStream_t s, size_t bytes, void** out) {
    std::lock_guard<std::mutex> lk(g_staging_mutex);
    Staging& st = g_staging[std::make_pair(dev, s)];
    if (st.bytes < bytes) {
        if (st.ptr) {
            if (cudaStreamSynchronize(s) != cudaSuccess || cudaFree(st.ptr) != cudaSuccess) {
                cudaGetLastError();
                return TG_ERR_LAUNCH;
            }
            st.ptr = nullptr;
            st.bytes = 0;
        }
        if (cudaMalloc(&st.ptr, bytes) != cudaSuccess) {
            cudaGetLastError();
            st.ptr = nullptr;
            return TG_ERR_NO_MEMORY;
        }
        st.bytes = bytes;
    }
    *out = st.ptr;
    return TG_OK;
}

// Copy a rows×cols matrix of `elem_bytes` (2 or 4) byte elements.
tg_status_t copy_matrix(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows,
                        int64_t cols, int elem_bytes, int num_sms, cudaStream_t s) {
    const int64_t steps = rows * ((cols + 255) / 256);  // warp steps of 256 elements
    const int64_t blocks = (steps + 7) / 8;             // 8 warps per block
    const unsigned grid = static_cast<unsigned>(blocks < 8 * num_sms ? blocks : 8 * num_sms);
    // A plain launch: it starts once the previous kernel has completed (as a
    // dependent launch its many small CTAs sat on the SMs beside the previous
    // GEMM and slowed it).  It lets the next kernel launch early.
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    const cudaError_t e =
        elem_bytes == 4
            ? cudaLaunchKernelEx(&cfg, tg::tg_copy_matrix<uint32_t>,
                                 static_cast<const uint32_t*>(src), ld_src,
                                 static_cast<uint32_t*>(dst), ld_dst, rows, cols)
            : cudaLaunchKernelEx(&cfg, tg::tg_copy_matrix<uint16_t>,
                                 static_cast<const uint16_t*>(src), ld_src,
                                 static_cast<uint16_t*>(dst), ld_dst, rows, cols);
    if (e != cudaSuccess) cudaGetLastError();
    return e == cudaSuccess ? TG_OK : TG_ERR_LAUNCH;
}

// Launch the planned kernel for operands in the tensor memory-access layout.
template <typename T>
tg_status_t launch_planned(tg_plan_t pl, const void* A, const void* B, void* C, int64_t M,
                           int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                           const tg::EpilogueSpec& ep, cudaStream_t s, int dev, DeviceState* ds) {
    switch (pl.kernel) {
        case TG_KERNEL_PERSISTENT:
            if (pl.cluster == 2)
                return launch_pair<T>(A, B, C, pl, M, N, K, lda, ldb, ldc, ep, s, dev, ds);
            if (pl.bn == kBigBN)
                return launch_persistent<kBigBN, kBigStages, T>(A, B, C, pl, M, N, K, lda, ldb,
                                                               ldc, ep, s);
            if (pl.bn == kSmallBN)
                return launch_persistent<kSmallBN, kSmallStages, T>(A, B, C, pl, M, N, K, lda,
                                                                   ldb, ldc, ep, s);
            return launch_persistent<kMidBN, kMidStages, T>(A, B, C, pl, M, N, K, lda, ldb, ldc,
                                                           ep, s);
        case TG_KERNEL_SKINNY: {
            const uint64_t timeout = g_timeout_ns.load();
            const int32_t inject = g_inject.exchange(0);
            record_launch(pl, pl.grid, pl.split_k, pl.cluster);
            return tg::skinny_launch<T>(A, B, C, pl, M, N, K, lda, ldb, ldc, ep, s, dev,
                                        ds->num_sms, timeout, inject, encode_2d);
        }
        default:
            return TG_ERR_INVALID_VALUE;
    }
}

// C = out(act(A·B + bias) + R) for 16-bit input type T (__half or
// __nv_bfloat16): plan, stage operands the tensor memory-access unit cannot
// address, launch the planned kernel on `stream`, and copy a staged C back.
// Arguments were validated by the caller.
template <typename T>
tg_status_t gemm_impl(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc, const tg::EpilogueSpec& ep,
                      void* stream) {
    if (M == 0 || N == 0) return TG_OK;
    int dev = 0;
    DeviceState* ds = nullptr;
    tg_status_t st = current_device(&dev, &ds);
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    tg_plan_t pl;
    const PlanLimits lim = device_limits(*ds);
    st = plan_limited(M, N, K, lim, &pl);
    if (st != TG_OK) return st;
    apply_forced_config(M, N, K, lim, &pl);

    if (pl.kernel == TG_KERNEL_FILL) {
        record_launch(pl, pl.grid, pl.split_k, pl.cluster);
        if (ep.e.bias == nullptr && ep.e.resid == nullptr && !ep.out_f32) {
            // +0 has the same (all-zero) bits in fp16 and bf16; any ldc works
            tg::tg_fill_zero_f16<<<static_cast<unsigned>(pl.grid), 256, 0, s>>>(
                static_cast<__half*>(C), M, N, ldc);
        } else {
            tg::tg_epilogue_only<T><<<static_cast<unsigned>(pl.grid), 256, 0, s>>>(
                C, ldc, ep.out_f32, ep.e, ep.relu, M, N);
        }
        return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_LAUNCH;
    }
    // C's element size and the tensor memory-access layout rule for it:
    // 16-byte aligned rows, i.e. ldc a multiple of 16 / elem_c.
    const int elem_c = ep.out_f32 ? 4 : 2;
    const bool a_ok = tma_layout_ok(A, lda), b_ok = tma_layout_ok(B, ldb);
    const bool c_ok = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && (ldc * elem_c) % 16 == 0;
    if (a_ok && b_ok && c_ok)
        return launch_planned<T>(pl, A, B, C, M, N, K, lda, ldb, ldc, ep, s, dev, ds);

    // Staging: aligned copies with leading dimensions rounded up to 8.
    const int64_t lda2 = a_ok ? lda : round_up8(K), ldb2 = b_ok ? ldb : round_up8(N);
    const int64_t ldc2 = c_ok ? ldc : round_up8(N);
    auto align256 = [](int64_t b) { return (b + 255) / 256 * 256; };
    const int64_t bytes_a = a_ok ? 0 : align256(M * lda2 * 2);
    const int64_t bytes_b = b_ok ? 0 : align256(K * ldb2 * 2);
    const int64_t bytes_c = c_ok ? 0 : align256(M * ldc2 * elem_c);
    void* buf = nullptr;
    st = staging_buffer(dev, s, static_cast<size_t>(bytes_a + bytes_b + bytes_c), &buf);
    if (st != TG_OK) return st;
    char* p = static_cast<char*>(buf);
    const void* A2 = a_ok ? A : p;
    const void* B2 = b_ok ? B : p + bytes_a;
    void* C2 = c_ok ? C : p + bytes_a + bytes_b;
    if (!a_ok && (st = copy_matrix(A, lda, p, lda2, M, K, 2, ds->num_sms, s)) != TG_OK) return st;
    if (!b_ok && (st = copy_matrix(B, ldb, p + bytes_a, ldb2, K, N, 2, ds->num_sms, s)) != TG_OK)
        return st;
    st = launch_planned<T>(pl, A2, B2, C2, M, N, K, lda2, ldb2, ldc2, ep, s, dev, ds);
    if (st != TG_OK || c_ok) return st;
    return copy_matrix(C2, ldc2, C, ldc, M, N, elem_c, ds->num_sms, s);
}

tg::EpilogueSpec plain_epilogue(int epilogue) {
    tg::EpilogueSpec ep;
    ep.relu = epilogue == TG_EPI_RELU ? 1 : 0;
    return ep;
}

// tg_gemm_ex's own argument checks (beyond validate): types, the residual's
// stride and the alignment of bias, residual and an fp32 C.
tg_status_t validate_ex(int32_t in_dtype, const void* C, int64_t M, int64_t N,
                        const tg_epilogue_ex_t& x) {
    if (in_dtype != TG_DTYPE_F16 && in_dtype != TG_DTYPE_BF16) return TG_ERR_INVALID_VALUE;
    if (x.out_dtype != in_dtype && x.out_dtype != TG_DTYPE_F32) return TG_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return TG_OK;
    if (x.residual != nullptr && x.ldr < N) return TG_ERR_INVALID_VALUE;
    if (x.bias != nullptr && (reinterpret_cast<uintptr_t>(x.bias) & 3u) != 0)
        return TG_ERR_MISALIGNED;
    if (x.residual != nullptr && (reinterpret_cast<uintptr_t>(x.residual) & 1u) != 0)
        return TG_ERR_MISALIGNED;
    if (x.out_dtype == TG_DTYPE_F32 && (reinterpret_cast<uintptr_t>(C) & 3u) != 0)
        return TG_ERR_MISALIGNED;
    return TG_OK;
}

// Per-(device, stream) fp16 buffer for dequantised MXFP4 weights (M > 128
// path); grown on demand like the staging buffer.
std::mutex g_deq_mutex;
std::map<std::pair<int, cudaStream_t>, Staging> g_deq;

tg_status_t dequant_buffer(int dev, cudaStream_t s, size_t bytes, void** out) {
    std::lock_guard<std::mutex> lk(g_deq_mutex);
    Staging& st = g_deq[std::make_pair(dev, s)];
    if (st.bytes < bytes) {
        if (st.ptr) {
            if (cudaStreamSynchronize(s) != cudaSuccess || cudaFree(st.ptr) != cudaSuccess) {
                cudaGetLastError();
                return TG_ERR_LAUNCH;
            }
            st.ptr = nullptr;
            st.bytes = 0;
        }
        if (cudaMalloc(&st.ptr, bytes) != cudaSuccess) {
            cudaGetLastError();
            st.ptr = nullptr;
            return TG_ERR_NO_MEMORY;
        }
        st.bytes = bytes;
    }
    *out = st.ptr;
    return TG_OK;
}

// Whether TGEMM_FORCE_CFG names one of the dense tile kernels (the MXFP4
// entry point then takes its dequantise-then-GEMM path even for M <= 128).
bool forced_dense_kernel() {
    const char* f = std::getenv("TGEMM_FORCE_CFG");
    return f != nullptr && (std::strcmp(f, "pair256") == 0 ||
                            std::strcmp(f, "persistent256") == 0 ||
                            std::strcmp(f, "persistent128") == 0 ||
                            std::strcmp(f, "persistent64") == 0);
}

// 2:4 sparse A: tensor maps, kernel choice, tile plan and launch (operands in
// the tensor memory-access layout, checked by the caller).  The kernel is
// tg::sp24_use_pairs' choice (sparse_plan.h).
// TGEMM_FORCE_SP24 = pair | cta overrides the choice (tests and sweeps).  Both kernels take the same tensor maps: per CTA 128 rows of
// Ac and E and 128 k of B per stage.
template <typename T>
tg_status_t launch_sp24(const void* Ac, const void* E, const void* B, void* C, int64_t M,
                        int64_t N, int64_t K, int64_t ldac, int64_t lde, int64_t ldb,
                        int64_t ldc, const tg::EpilogueSpec& ep, cudaStream_t s,
                        DeviceState* ds) {
    using Cfg = tg::SparseCfg;
    using PairCfg = tg::SparsePairCfg<kSpPairStages>;
    static_assert(PairCfg::BK == Cfg::BK && PairCfg::BM == 2 * Cfg::BM,
                  "the two sparse kernels share their tensor maps");
    constexpr CUtensorMapDataType dt = tensor_map_type<T>();
    CUtensorMap tmA, tmB, tmE, tmC;
    if (!encode_2d(&tmA, Ac, K / 2, M, ldac * 2, 64, Cfg::BM, dt) ||
        !encode_2d(&tmB, B, N, K, ldb * 2, 64, Cfg::BK, dt) ||
        !encode_2d_sw(&tmE, E, K / 32, M, lde * 4, Cfg::BK / 32, Cfg::BM,
                      CU_TENSOR_MAP_DATA_TYPE_UINT32, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !(ep.out_f32 ? encode_2d(&tmC, C, N, M, ldc * 4, 32, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32)
                     : encode_2d(&tmC, C, N, M, ldc * 2, 64, 32, dt)))
        return TG_ERR_LAUNCH;
    static_assert(PairCfg::BN == 256 && Cfg::BN == 128, "the tile sizes sparse_plan.h assumes");
    bool pair = tg::sp24_use_pairs(M, N, K, ds->max_sp_pairs, ds->num_sms);
    if (const char* f = std::getenv("TGEMM_FORCE_SP24")) {
        if (std::strcmp(f, "pair") == 0) pair = ds->max_sp_pairs >= 1;
        if (std::strcmp(f, "cta") == 0) pair = false;
    }
    const int64_t bm = pair ? PairCfg::BM : Cfg::BM;
    const int64_t bn = pair ? PairCfg::BN : Cfg::BN;
    tg::SparseParams sp;
    tg::PersistentParams& prm = sp.base;
    prm.M = static_cast<int32_t>(M);
    prm.N = static_cast<int32_t>(N);
    prm.K = static_cast<int32_t>(K);
    prm.tiles_m = static_cast<int32_t>(ceil_div(M, bm));
    prm.tiles_n = static_cast<int32_t>(ceil_div(N, bn));
    prm.num_tiles = prm.tiles_m * prm.tiles_n;
    prm.k_blocks = static_cast<int32_t>(ceil_div(K, Cfg::BK));
    prm.group_m = prm.tiles_m < 16 ? prm.tiles_m : 16;
    prm.relu = ep.relu;
    prm.inject = g_inject.exchange(0);
    prm.timeout_ns = g_timeout_ns.load();
    prm.e = ep.e;
    prm.out_f32 = ep.out_f32;
    sp.words = static_cast<int32_t>(K / 32);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    tg::set_dependent_launch(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (pair) {
        const int64_t pairs = prm.num_tiles < ds->max_sp_pairs ? prm.num_tiles : ds->max_sp_pairs;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
        cfg.blockDim = dim3(PairCfg::kThreads);
        cfg.numAttrs = 2;
        if (ep.e.bias == nullptr && ep.e.resid == nullptr && ep.out_f32 == 0) {
            cfg.dynamicSmemBytes = tg::SparsePairCfg<kSpPairStagesPlain>::kSmemBytes;
            e = cudaLaunchKernelEx(&cfg, tg::tg_gemm_sp24_pair<kSpPairStagesPlain, T, false>, tmA,
                                   tmB, tmE, tmC, sp);
        } else {
            cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
            e = cudaLaunchKernelEx(&cfg, tg::tg_gemm_sp24_pair<kSpPairStages, T, true>, tmA, tmB,
                                   tmE, tmC, sp);
        }
    } else {
        const int64_t grid = prm.num_tiles < ds->num_sms ? prm.num_tiles : ds->num_sms;
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(Cfg::kThreads);
        cfg.dynamicSmemBytes = Cfg::kSmemBytes;
        e = (ep.e.bias == nullptr && ep.e.resid == nullptr && ep.out_f32 == 0)
                ? cudaLaunchKernelEx(&cfg, tg::tg_gemm_sp24<T, false>, tmA, tmB, tmE, tmC, sp)
                : cudaLaunchKernelEx(&cfg, tg::tg_gemm_sp24<T>, tmA, tmB, tmE, tmC, sp);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    return TG_OK;
}

// The plan tg_gemm_f16 launches, within the limits of a device.
tg_status_t plan_limited(int64_t M, int64_t N, int64_t K, const PlanLimits& lim,
                         tg_plan_t* plan) {
    const int32_t num_sms = lim.num_sms;
    if (plan == nullptr || num_sms < 1) return TG_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return TG_ERR_INVALID_VALUE;
    std::memset(plan, 0, sizeof(*plan));
    if (M == 0 || N == 0) {
        plan->kernel = TG_KERNEL_NONE;
        return TG_OK;
    }
    if (K == 0) {
        plan->kernel = TG_KERNEL_FILL;
        plan->threads = 256;
        int64_t blocks = ceil_div(M * N, 256);
        plan->grid = blocks < 4 * num_sms ? blocks : 4 * num_sms;
        return TG_OK;
    }
    if (tg::skinny_applies(M, N, K)) {
        tg::skinny_plan(M, N, K, num_sms, plan);
        // clusters of a tile's four k-pieces only if all of them fit at once
        // (a second round of clusters would double the time)
        if (plan->cluster == 4 && plan->grid / 4 > lim.quads[plan->mma_n > 64 ? 1 : 0])
            plan->cluster = 1;
        return TG_OK;
    }
    // At least one full wave of 256×256 tiles on CTA pairs: the pair kernel.
    const int64_t tiles_pair = ceil_div(M, 256) * ceil_div(N, 256);
    if (lim.pairs >= 1 && tiles_pair >= lim.pairs) {
        plan_pair(M, N, K, lim.pairs, plan);
        return TG_OK;
    }
    // Less than a wave of pair tiles, but more 128×128 tiles than SMs (one-CTA
    // tiles would take two or more rounds) and K of at least 1024: one round of
    // pair tiles on part of the GPU still wins, since one-CTA 128×128 tiles run
    // at about 0.6 of the pair kernel's rate per SM.  Measured on GB300:
    // 2048×2048×8192 47 µs against 84 µs, 2048×1536×4096 26 µs against 42 µs,
    // 2048×2048×1024 14.1 µs against 16.4 µs.  With shorter K the pair kernel's
    // longer pipeline fill loses (2048×2048×256: 10.3 µs against 8.3 µs).
    const int64_t tiles128 = ceil_div(M, 128) * ceil_div(N, 128);
    if (lim.pairs >= 1 && tiles128 > num_sms && K >= 1024) {
        plan_pair(M, N, K, lim.pairs, plan);
        return TG_OK;
    }
    // 128×128 tiles would fill at most half the SMs: 128×64 tiles instead.
    // Timed from CUDA graphs against 128×128 on GB300 (same bits): 256^3
    // 3.89 -> 3.26 us, 512^3 5.32 -> 4.41, 1024^3 ReLU 7.32 -> 6.61,
    // 1024×1024×4096 18.2 -> 15.9.
    if (tiles128 * 2 <= num_sms) {
        plan_persistent(M, N, K, num_sms, kSmallBN, kSmallStages,
                        tg::PersistentCfg<kSmallBN, kSmallStages>::kSmemBytes, plan);
        return TG_OK;
    }
    const int64_t tiles256 = ceil_div(M, 128) * ceil_div(N, kBigBN);
    if (tiles256 >= num_sms || N <= kMidBN) {
        if (N <= kMidBN)
            plan_persistent(M, N, K, num_sms, kMidBN, kMidStages,
                            tg::PersistentCfg<kMidBN, kMidStages>::kSmemBytes, plan);
        else
            plan_persistent(M, N, K, num_sms, kBigBN, kBigStages,
                            tg::PersistentCfg<kBigBN, kBigStages>::kSmemBytes, plan);
    } else {
        plan_persistent(M, N, K, num_sms, kMidBN, kMidStages,
                        tg::PersistentCfg<kMidBN, kMidStages>::kSmemBytes, plan);
    }
    return TG_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

int64_t tg_ring_bytes(int32_t bm, int32_t bn, int32_t bk, int32_t stages, int32_t elem_bytes) {
    if (bm <= 0 || bn <= 0 || bk <= 0 || stages <= 0 || elem_bytes <= 0) return -1;
    const int64_t per_stage = (static_cast<int64_t>(bm) * bk + static_cast<int64_t>(bk) * bn) *
                              elem_bytes;
    return per_stage * stages;
}

tg_status_t tg_plan_f16(int64_t M, int64_t N, int64_t K, int32_t num_sms, tg_plan_t* plan) {
    if (num_sms < 1) return TG_ERR_INVALID_VALUE;
    return plan_limited(M, N, K, nominal_limits(num_sms), plan);
}

tg_status_t tg_plan_f16_limits(int64_t M, int64_t N, int64_t K, int32_t num_sms,
                               int32_t max_pairs, int32_t max_quads_narrow,
                               int32_t max_quads_wide, tg_plan_t* plan) {
    if (num_sms < 1 || max_pairs < 0 || max_quads_narrow < 0 || max_quads_wide < 0)
        return TG_ERR_INVALID_VALUE;
    PlanLimits l;
    l.num_sms = num_sms;
    l.pairs = max_pairs < num_sms / 2 ? max_pairs : num_sms / 2;
    l.quads[0] = max_quads_narrow;
    l.quads[1] = max_quads_wide;
    return plan_limited(M, N, K, l, plan);
}

tg_status_t tg_device_limits(int32_t* num_sms, int32_t* max_pairs, int32_t* max_quads_narrow,
                             int32_t* max_quads_wide) {
    if (num_sms == nullptr || max_pairs == nullptr || max_quads_narrow == nullptr ||
        max_quads_wide == nullptr)
        return TG_ERR_INVALID_VALUE;
    int dev = 0;
    DeviceState* ds = nullptr;
    const tg_status_t st = current_device(&dev, &ds);
    if (st != TG_OK) return st;
    *num_sms = ds->num_sms;
    *max_pairs = ds->max_pairs;
    *max_quads_narrow = ds->max_skinny_quads[0];
    *max_quads_wide = ds->max_skinny_quads[1];
    return TG_OK;
}

tg_status_t tg_debug_last_launch(tg_plan_t* plan) {
    if (plan == nullptr) return TG_ERR_INVALID_VALUE;
    *plan = g_last_launch;
    return TG_OK;
}

void tg_debug_map_cache_stats(uint64_t* hits, uint64_t* misses) {
    if (hits != nullptr) *hits = g_map_hits.load();
    if (misses != nullptr) *misses = g_map_misses.load();
}


tg_status_t tg_tile_coord(const tg_plan_t* plan, int64_t tile, int64_t* m_blk, int64_t* n_blk) {
    if (plan == nullptr || m_blk == nullptr || n_blk == nullptr) return TG_ERR_INVALID_VALUE;
    if (plan->kernel != TG_KERNEL_PERSISTENT || tile < 0 || tile >= plan->num_tiles)
        return TG_ERR_INVALID_VALUE;
    const tg::TileCoord c =
        tg::tile_coord(static_cast<int32_t>(tile), static_cast<int32_t>(plan->tiles_m),
                       static_cast<int32_t>(plan->tiles_n), plan->group_m);
    *m_blk = c.m_blk;
    *n_blk = c.n_blk;
    return TG_OK;
}

void tg_debug_set_wait_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns == 0 ? kDefaultTimeoutNs : ns);
}

void tg_debug_inject(int32_t mode) { g_inject.store(mode); }

const char* tg_status_string(tg_status_t s) {
    switch (s) {
        case TG_OK: return "TG_OK";
        case TG_ERR_INVALID_VALUE: return "TG_ERR_INVALID_VALUE";
        case TG_ERR_MISALIGNED: return "TG_ERR_MISALIGNED";
        case TG_ERR_UNSUPPORTED_DEVICE: return "TG_ERR_UNSUPPORTED_DEVICE";
        case TG_ERR_LAUNCH: return "TG_ERR_LAUNCH";
        case TG_ERR_NO_MEMORY: return "TG_ERR_NO_MEMORY";
        case TG_ERR_TIMEOUT: return "TG_ERR_TIMEOUT";
    }
    return "TG_ERR_UNKNOWN";
}

const char* tg_version(void) { return "libtgemm 0.1.0 (sm_103a)"; }

tg_status_t tg_gemm_f16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldc, int epilogue, void* stream) {
    const tg_status_t st = validate(A, B, C, M, N, K, lda, ldb, ldc, epilogue, false);
    if (st != TG_OK) return st;
    return gemm_impl<__half>(A, B, C, M, N, K, lda, ldb, ldc, plain_epilogue(epilogue), stream);
}

tg_status_t tg_gemm_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                         int64_t lda, int64_t ldb, int64_t ldc, int epilogue, void* stream) {
    const tg_status_t st = validate(A, B, C, M, N, K, lda, ldb, ldc, epilogue, false);
    if (st != TG_OK) return st;
    return gemm_impl<__nv_bfloat16>(A, B, C, M, N, K, lda, ldb, ldc, plain_epilogue(epilogue),
                                    stream);
}

tg_status_t tg_gemm_ex(int32_t in_dtype, const void* A, const void* B, void* C, int64_t M,
                       int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                       const tg_epilogue_ex_t* epi, void* stream) {
    tg_epilogue_ex_t x;
    if (epi != nullptr) {
        x = *epi;
    } else {
        std::memset(&x, 0, sizeof(x));
        x.activation = TG_EPI_NONE;
        x.out_dtype = in_dtype;
    }
    tg_status_t st = validate(A, B, C, M, N, K, lda, ldb, ldc, x.activation, false);
    if (st != TG_OK) return st;
    st = validate_ex(in_dtype, C, M, N, x);
    if (st != TG_OK) return st;
    tg::EpilogueSpec ep = plain_epilogue(x.activation);
    ep.out_f32 = x.out_dtype == TG_DTYPE_F32 ? 1 : 0;
    ep.e.bias = x.bias;
    ep.e.resid = x.residual;
    ep.e.ldr = x.residual != nullptr ? x.ldr : 0;
    ep.e.bias_vec = (reinterpret_cast<uintptr_t>(x.bias) & 15u) == 0 ? 1 : 0;
    ep.e.resid_vec =
        (reinterpret_cast<uintptr_t>(x.residual) & 15u) == 0 && (x.ldr & 7) == 0 ? 1 : 0;
    if (in_dtype == TG_DTYPE_BF16)
        return gemm_impl<__nv_bfloat16>(A, B, C, M, N, K, lda, ldb, ldc, ep, stream);
    return gemm_impl<__half>(A, B, C, M, N, K, lda, ldb, ldc, ep, stream);
}

tg_status_t tg_gemm_mxfp4(const void* A, const void* Bq, const void* Bscale, void* C, int64_t M,
                          int64_t N, int64_t K, int64_t lda, int64_t ldbq, int64_t ldbs,
                          int64_t ldc, const tg_epilogue_ex_t* epi, void* stream) {
    tg_epilogue_ex_t x;
    if (epi != nullptr) {
        x = *epi;
    } else {
        std::memset(&x, 0, sizeof(x));
        x.activation = TG_EPI_NONE;
        x.out_dtype = TG_DTYPE_F16;
    }
    if (x.activation != TG_EPI_NONE && x.activation != TG_EPI_RELU) return TG_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return TG_ERR_INVALID_VALUE;
    tg_status_t st = validate_ex(TG_DTYPE_F16, C, M, N, x);
    if (st != TG_OK || M == 0 || N == 0) return st;
    if (C == nullptr || ldc < N) return TG_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(C) & 1u) != 0) return TG_ERR_MISALIGNED;
    if (K > 0) {
        if (A == nullptr || Bq == nullptr || Bscale == nullptr || lda < K ||
            ldbq < (K + 1) / 2 || ldbs < N)
            return TG_ERR_INVALID_VALUE;
        if ((reinterpret_cast<uintptr_t>(A) & 1u) != 0 ||
            (reinterpret_cast<uintptr_t>(Bq) & 15u) != 0 ||
            (reinterpret_cast<uintptr_t>(Bscale) & 15u) != 0 || (ldbq & 15) != 0 ||
            (ldbs & 15) != 0)
            return TG_ERR_MISALIGNED;
    }
    int dev = 0;
    DeviceState* ds = nullptr;
    st = current_device(&dev, &ds);
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    tg::EpilogueSpec ep = plain_epilogue(x.activation);
    ep.out_f32 = x.out_dtype == TG_DTYPE_F32 ? 1 : 0;
    ep.e.bias = x.bias;
    ep.e.resid = x.residual;
    ep.e.ldr = x.residual != nullptr ? x.ldr : 0;
    ep.e.bias_vec = (reinterpret_cast<uintptr_t>(x.bias) & 15u) == 0 ? 1 : 0;
    ep.e.resid_vec =
        (reinterpret_cast<uintptr_t>(x.residual) & 15u) == 0 && (x.ldr & 7) == 0 ? 1 : 0;
    if (K == 0)  // the product is +0: only the epilogue remains
        return gemm_impl<__half>(nullptr, nullptr, C, M, N, 0, 0, 0, ldc, ep, stream);

    if (M <= 128 && !forced_dense_kernel()) {
        // Weight streaming: decode inside the split-K kernel.
        tg_plan_t pl;
        std::memset(&pl, 0, sizeof(pl));
        tg::skinny_mx_plan(M, N, K, ds->num_sms, &pl);
        const void* A2 = A;
        int64_t lda2 = lda;
        if (!tma_layout_ok(A, lda)) {  // A in the staging buffer, rows 16-byte aligned
            lda2 = round_up8(K);
            void* buf = nullptr;
            st = staging_buffer(dev, s, static_cast<size_t>(M * lda2 * 2), &buf);
            if (st != TG_OK) return st;
            if ((st = copy_matrix(A, lda, buf, lda2, M, K, 2, ds->num_sms, s)) != TG_OK) return st;
            A2 = buf;
        }
        return tg::skinny_mx_launch(A2, Bq, Bscale, C, pl, M, N, K, lda2, ldbq, ldbs, ldc, ep,
                                    s, dev, ds->num_sms, g_timeout_ns.load(),
                                    g_inject.exchange(0), encode_2d_sw);
    }
    // Compute-bound sizes: dequantise once to fp16, then the dense GEMM.
    const int64_t ldd = round_up8(N);
    void* deq = nullptr;
    st = dequant_buffer(dev, s, static_cast<size_t>(K * ldd * 2), &deq);
    if (st != TG_OK) return st;
    const int64_t tiles = ((K + 63) / 64) * ((N + 63) / 64);  // 64 × 64 per block iteration
    const unsigned grid = static_cast<unsigned>(tiles < 8 * ds->num_sms ? tiles : 8 * ds->num_sms);
    // A plain launch that lets the next kernel launch early (as a dependent
    // launch it slowed the previous kernel, like the staging copy).
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    if (cudaLaunchKernelEx(&cfg, tg::tg_mxfp4_dequant_f16, static_cast<const uint8_t*>(Bq), ldbq,
                           static_cast<const uint8_t*>(Bscale), ldbs, K, N,
                           static_cast<uint16_t*>(deq), ldd) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    return gemm_impl<__half>(A, deq, C, M, N, K, lda, ldd, ldc, ep, stream);
}

tg_status_t tg_gemm_sp24(int32_t in_dtype, const void* Ac, const void* E, const void* B, void* C,
                         int64_t M, int64_t N, int64_t K, int64_t ldac, int64_t lde, int64_t ldb,
                         int64_t ldc, const tg_epilogue_ex_t* epi, void* stream) {
    tg_epilogue_ex_t x;
    if (epi != nullptr) {
        x = *epi;
    } else {
        std::memset(&x, 0, sizeof(x));
        x.activation = TG_EPI_NONE;
        x.out_dtype = in_dtype;
    }
    if (x.activation != TG_EPI_NONE && x.activation != TG_EPI_RELU) return TG_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || (K % 32) != 0)
        return TG_ERR_INVALID_VALUE;
    tg_status_t st = validate_ex(in_dtype, C, M, N, x);
    if (st != TG_OK || M == 0 || N == 0) return st;
    if (C == nullptr || ldc < N) return TG_ERR_INVALID_VALUE;
    const int elem_c = x.out_dtype == TG_DTYPE_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(C) & 15u) != 0 || (ldc * elem_c) % 16 != 0)
        return TG_ERR_MISALIGNED;
    if (K > 0) {
        if (Ac == nullptr || E == nullptr || B == nullptr || ldac < K / 2 || lde < K / 32 ||
            ldb < N)
            return TG_ERR_INVALID_VALUE;
        if ((reinterpret_cast<uintptr_t>(Ac) & 15u) != 0 ||
            (reinterpret_cast<uintptr_t>(E) & 15u) != 0 ||
            (reinterpret_cast<uintptr_t>(B) & 15u) != 0 || (ldac & 7) != 0 || (lde & 3) != 0 ||
            (ldb & 7) != 0)
            return TG_ERR_MISALIGNED;
    }
    int dev = 0;
    DeviceState* ds = nullptr;
    st = current_device(&dev, &ds);
    if (st != TG_OK) return st;
    tg::EpilogueSpec ep = plain_epilogue(x.activation);
    ep.out_f32 = x.out_dtype == TG_DTYPE_F32 ? 1 : 0;
    ep.e.bias = x.bias;
    ep.e.resid = x.residual;
    ep.e.ldr = x.residual != nullptr ? x.ldr : 0;
    ep.e.bias_vec = (reinterpret_cast<uintptr_t>(x.bias) & 15u) == 0 ? 1 : 0;
    ep.e.resid_vec =
        (reinterpret_cast<uintptr_t>(x.residual) & 15u) == 0 && (x.ldr & 7) == 0 ? 1 : 0;
    if (K == 0) {
        if (in_dtype == TG_DTYPE_BF16)
            return gemm_impl<__nv_bfloat16>(nullptr, nullptr, C, M, N, 0, 0, 0, ldc, ep, stream);
        return gemm_impl<__half>(nullptr, nullptr, C, M, N, 0, 0, 0, ldc, ep, stream);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (in_dtype == TG_DTYPE_BF16)
        return launch_sp24<__nv_bfloat16>(Ac, E, B, C, M, N, K, ldac, lde, ldb, ldc, ep, s, ds);
    return launch_sp24<__half>(Ac, E, B, C, M, N, K, ldac, lde, ldb, ldc, ep, s, ds);
}

tg_status_t tg_sync_status(void* stream) {
    int dev = 0;
    DeviceState* ds = nullptr;
    tg_status_t st = current_device(&dev, &ds);
    if (st != TG_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    unsigned int flags = 0;
    if (cudaMemcpyFromSymbol(&flags, tg::g_wait_timeout_flags, sizeof(flags)) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    if (flags != 0) {
        // A kernel gave up early: let every queued kernel finish, then clear
        // the split-K counters it may have left non-zero before anything reuses them.
        cudaDeviceSynchronize();
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(tg::g_wait_timeout_flags, &zero, sizeof(zero));
        tg::splitk_reset_counters(dev);
        noalloc_reset_counters(dev);
        cudaGetLastError();
        return TG_ERR_TIMEOUT;
    }
    return TG_OK;
}

}  // extern "C"

// ====================================================================== host buffers in and out
//
// tg_gemm_f16_host: device copies of A, B and C plus two copy streams per
// (device, stream); see include/tgemm.h for the overlap scheme.

namespace {

constexpr int kHostMaxBlocks = 8;           // column blocks per call
constexpr int64_t kHostFirstBlockCols = 1024;  // then doubling, up to kHostMaxBlockCols
constexpr int64_t kHostMaxBlockCols = 8192;

struct HostPipeline {
    void* dA = nullptr;
    void* dB = nullptr;
    void* dC = nullptr;
    size_t bytes_a = 0, bytes_b = 0, bytes_c = 0;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t uploaded[kHostMaxBlocks] = {};
    cudaEvent_t computed[kHostMaxBlocks] = {};
    bool ready = false;
};

std::mutex g_host_mutex;
std::map<std::pair<int, cudaStream_t>, HostPipeline> g_host;

// Grow one device copy to `need` bytes.  Earlier calls on this pipeline may
// still read or write the old buffer: `stream` (which every call leaves
// waiting for its last download) is synchronised first.
tg_status_t host_buffer(void** p, size_t* have, size_t need, cudaStream_t stream) {
    if (*have >= need) return TG_OK;
    if (*p != nullptr) {
        if (cudaStreamSynchronize(stream) != cudaSuccess || cudaFree(*p) != cudaSuccess) {
            cudaGetLastError();
            return TG_ERR_LAUNCH;
        }
        *p = nullptr;
        *have = 0;
    }
    if (cudaMalloc(p, need) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return TG_ERR_NO_MEMORY;
    }
    *have = need;
    return TG_OK;
}

tg_status_t host_pipeline_init(HostPipeline& hp) {
    if (hp.ready) return TG_OK;
    bool ok = cudaStreamCreateWithFlags(&hp.up, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.down, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kHostMaxBlocks; ++i)
        ok = cudaEventCreateWithFlags(&hp.uploaded[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp.computed[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    hp.ready = true;
    return TG_OK;
}

}  // namespace

extern "C" tg_status_t tg_gemm_f16_host(const void* A, const void* B, void* C, int64_t M,
                                        int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                        int64_t ldc, int epilogue, void* stream) {
    tg_status_t st = validate(A, B, C, M, N, K, lda, ldb, ldc, epilogue, false);
    if (st != TG_OK || M == 0 || N == 0) return st;
    int dev = 0;
    DeviceState* ds = nullptr;
    st = current_device(&dev, &ds);
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lk(g_host_mutex);
    HostPipeline& hp = g_host[std::make_pair(dev, s)];
    if ((st = host_pipeline_init(hp)) != TG_OK) return st;
    // Device copies: row strides rounded up to 8 elements (16-byte rows).
    const int64_t Kp = round_up8(K), Np = round_up8(N);
    if ((st = host_buffer(&hp.dA, &hp.bytes_a, static_cast<size_t>(M * Kp * 2) + 16, s)) != TG_OK ||
        (st = host_buffer(&hp.dB, &hp.bytes_b, static_cast<size_t>(K * Np * 2) + 16, s)) != TG_OK ||
        (st = host_buffer(&hp.dC, &hp.bytes_c, static_cast<size_t>(M * Np * 2) + 16, s)) != TG_OK)
        return st;

    // Column blocks: a narrow first one, so that downloads start early, then
    // doubling widths (wider rows copy faster) up to kHostMaxBlockCols; the
    // last of at most kHostMaxBlocks takes the rest.  Every block but the
    // last is a multiple of 256 columns, so each block's device pointers stay
    // 16-byte aligned.
    int64_t c0s[kHostMaxBlocks + 1];
    int blocks = 0;
    {
        int64_t c = 0, w = kHostFirstBlockCols;
        while (c < N) {
            if (blocks == kHostMaxBlocks - 1 || w > N - c) w = N - c;
            c0s[blocks++] = c;
            c += w;
            w = w * 2 < kHostMaxBlockCols ? w * 2 : kHostMaxBlockCols;
        }
        c0s[blocks] = N;
    }

    const char* hA = static_cast<const char*>(A);
    const char* hB = static_cast<const char*>(B);
    char* hC = static_cast<char*>(C);
    char* dA = static_cast<char*>(hp.dA);
    char* dB = static_cast<char*>(hp.dB);
    char* dC = static_cast<char*>(hp.dC);
    const tg::EpilogueSpec ep = plain_epilogue(epilogue);
    auto fail = [] {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    };

    // Everything already on `stream` (earlier calls' products included)
    // comes before this call's uploads overwrite the device copies.
    if (cudaEventRecord(hp.start, s) != cudaSuccess ||
        cudaStreamWaitEvent(hp.up, hp.start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp.down, hp.start, 0) != cudaSuccess)
        return fail();
    if (K > 0 && cudaMemcpy2DAsync(dA, Kp * 2, hA, lda * 2, K * 2, M, cudaMemcpyHostToDevice,
                                   hp.up) != cudaSuccess)
        return fail();
    for (int j = 0; j < blocks; ++j) {
        const int64_t c0 = c0s[j];
        const int64_t w = c0s[j + 1] - c0;
        if (K > 0 && cudaMemcpy2DAsync(dB + c0 * 2, Np * 2, hB + c0 * 2, ldb * 2, w * 2, K,
                                       cudaMemcpyHostToDevice, hp.up) != cudaSuccess)
            return fail();
        if (cudaEventRecord(hp.uploaded[j], hp.up) != cudaSuccess ||
            cudaStreamWaitEvent(s, hp.uploaded[j], 0) != cudaSuccess)
            return fail();
        st = gemm_impl<__half>(dA, dB + c0 * 2, dC + c0 * 2, M, w, K, Kp, Np, Np, ep, s);
        if (st != TG_OK) return st;
        if (cudaEventRecord(hp.computed[j], s) != cudaSuccess ||
            cudaStreamWaitEvent(hp.down, hp.computed[j], 0) != cudaSuccess ||
            cudaMemcpy2DAsync(hC + c0 * 2, ldc * 2, dC + c0 * 2, Np * 2, w * 2, M,
                              cudaMemcpyDeviceToHost, hp.down) != cudaSuccess)
            return fail();
    }
    if (cudaEventRecord(hp.done, hp.down) != cudaSuccess ||
        cudaStreamWaitEvent(s, hp.done, 0) != cudaSuccess)
        return fail();
    return TG_OK;
}

// ====================================================================== no-allocation variant
//
// tg_gemm_f16_noalloc runs the skinny split-K kernel with its scratch (fp32
// partial sums and the per-warp piece counters) in the file-scope array below
// instead of a workspace obtained from cudaMalloc.  It serves callers that
// cannot allocate device memory at call time.  The array is a fixed
// TG_NOALLOC_SCRATCH_BYTES; every device that loads this library holds it
// until the process exits.
//
// In host code `g_noalloc_scratch` only names the variable: it is not a
// device address.  Its device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed to the kernel.

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TG_NOALLOC_SCRATCH_BYTES];

// Counter words first (4 per CTA, 16 bytes), then the fp32 partial slots
// (two per CTA).
constexpr int64_t kNoallocCounterBytes = 64 * 1024;
constexpr int64_t kNoallocMaxCtas = kNoallocCounterBytes / 16;

struct NoallocDeviceState {
    bool ready = false;
    unsigned char* base = nullptr;  // device address of g_noalloc_scratch
};

std::mutex g_noalloc_mutex;
NoallocDeviceState g_noalloc[kMaxDevices];

// After a timed-out launch: clear the counter words (the device is idle).
void noalloc_reset_counters(int dev) {
    std::lock_guard<std::mutex> lk(g_noalloc_mutex);
    if (dev >= 0 && dev < kMaxDevices && g_noalloc[dev].ready)
        cudaMemset(g_noalloc[dev].base, 0, kNoallocCounterBytes);
}

}  // namespace

extern "C" tg_status_t tg_gemm_f16_noalloc(const void* A, const void* B, void* C, int64_t M,
                                           int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                           int64_t ldc, int epilogue, void* stream) {
    tg_status_t st = validate(A, B, C, M, N, K, lda, ldb, ldc, epilogue);
    if (st != TG_OK || M == 0 || N == 0) return st;
    if (M > 128) return TG_ERR_INVALID_VALUE;  // the split-K kernel covers M <= 128 only
    int dev = 0;
    DeviceState* ds = nullptr;
    st = current_device(&dev, &ds);
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (K == 0) {  // C = epi(0): no scratch involved
        tg_plan_t pf;
        tg_plan_f16(M, N, K, ds->num_sms, &pf);
        tg::tg_fill_zero_f16<<<static_cast<unsigned>(pf.grid), 256, 0, s>>>(
            static_cast<__half*>(C), M, N, ldc);
        return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_LAUNCH;
    }

    tg_plan_t pl;
    if ((st = plan_limited(M, N, K, device_limits(*ds), &pl)) != TG_OK) return st;
    if (pl.kernel != TG_KERNEL_SKINNY) return TG_ERR_INVALID_VALUE;
    if (pl.grid > kNoallocMaxCtas ||
        kNoallocCounterBytes + 2 * pl.grid * tg::kSkSlotFloats * 4 > TG_NOALLOC_SCRATCH_BYTES)
        return TG_ERR_INVALID_VALUE;  // would need more scratch than the array holds

    tg::SkinnyParams prm;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mutex);
        NoallocDeviceState& ns = g_noalloc[dev];
        if (!ns.ready) {
            // Once per device, with that device current: the array's device
            // address, and the counter words cleared (each launch then leaves
            // them at zero: the warp that sums a tile zeroes its counter).
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return TG_ERR_LAUNCH;
            }
            if (cudaMemsetAsync(p, 0, kNoallocCounterBytes, s) != cudaSuccess) {
                cudaGetLastError();
                return TG_ERR_LAUNCH;
            }
            ns.base = static_cast<unsigned char*>(p);
            ns.ready = true;
        }
        prm.counters = reinterpret_cast<uint32_t*>(ns.base);
        prm.ws = reinterpret_cast<float*>(ns.base + kNoallocCounterBytes);
    }

    const int64_t Mp = pl.mma_n;
    CUtensorMap tmA, tmB;
    // B boxes: 64 columns × the plan's k per unit (the kernel arms its
    // barriers for that many rows)
    if (!encode_2d(&tmB, B, N, K, ldb * 2, 64, static_cast<uint32_t>(pl.bk),
                   CU_TENSOR_MAP_DATA_TYPE_FLOAT16) ||
        !encode_2d(&tmA, A, K, M, lda * 2, 64, static_cast<uint32_t>(Mp),
                   CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
        return TG_ERR_LAUNCH;
    prm.M = static_cast<int32_t>(M);
    prm.N = static_cast<int32_t>(N);
    prm.K = static_cast<int32_t>(K);
    prm.Mp = static_cast<int32_t>(Mp);
    prm.tiles_n = static_cast<int32_t>(pl.tiles_n);
    prm.k_blocks = static_cast<int32_t>(pl.k_blocks);
    prm.total_units = pl.tiles_n * pl.k_blocks;
    prm.relu = epilogue == TG_EPI_RELU ? 1 : 0;
    prm.inject = 0;
    prm.timeout_ns = g_timeout_ns.load();
    prm.C = C;
    prm.ldc = ldc;

    record_launch(pl, pl.grid, pl.split_k, pl.cluster);
    if (tg::skinny_launch_kernel<__half>(tmB, tmA, prm, pl.grid, s, pl.cluster) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_LAUNCH;
    }
    return TG_OK;
}
