// launch_util.cu -- per-device launch facts, shared-memory opt-ins and the TMA
// tensor-map cache (see launch_util.h).
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "launch_table.h"
#include "launch_util.h"

namespace ck {
namespace {

constexpr int kMaxDevices = 64;

std::atomic<int> g_sms[kMaxDevices];  // 0 = not looked up yet

// (device, kernel) pairs whose shared-memory opt-in is done (a few dozen
// kernels at most), and occupancy per (device, kernel, threads, smem)
OnceTable<const void *, 512> g_optins;
struct OccKey {
    const void *kernel;
    int threads;
    size_t smem;
    bool operator==(const OccKey &o) const {
        return kernel == o.kernel && threads == o.threads && smem == o.smem;
    }
};
ValueCache<OccKey, int, 256> g_occ;
struct ClusterKey {
    const void *kernel;
    int threads;
    size_t smem;
    int cluster;
    bool operator==(const ClusterKey &o) const {
        return kernel == o.kernel && threads == o.threads && smem == o.smem && cluster == o.cluster;
    }
};
ValueCache<ClusterKey, int, 64> g_clusters;

// Tensor-map cache: direct-mapped on a hash of the request.
struct MapKey {
    const void *ptr;
    int64_t rows, cols;
    int dtype, elem_bytes, box_cols, box_rows, swizzle;
    bool operator==(const MapKey &o) const {
        return ptr == o.ptr && rows == o.rows && cols == o.cols && dtype == o.dtype &&
               elem_bytes == o.elem_bytes && box_cols == o.box_cols && box_rows == o.box_rows &&
               swizzle == o.swizzle;
    }
};
struct MapSlot {
    bool used;
    MapKey key;
    CUtensorMap map;
};
constexpr int kMapSlots = 1024;
std::mutex g_map_mu;
MapSlot g_maps[kMapSlots];
uint64_t g_map_hits = 0, g_map_misses = 0;

uint64_t mix(uint64_t h, uint64_t v) {
    h ^= v + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    return h;
}

size_t slot_of(const MapKey &k) {
    uint64_t h = reinterpret_cast<uintptr_t>(k.ptr);
    h = mix(h, static_cast<uint64_t>(k.rows));
    h = mix(h, static_cast<uint64_t>(k.cols));
    h = mix(h, static_cast<uint64_t>(k.dtype) << 32 | static_cast<uint32_t>(k.elem_bytes));
    h = mix(h, static_cast<uint64_t>(k.box_cols) << 32 | static_cast<uint32_t>(k.box_rows));
    h = mix(h, static_cast<uint64_t>(k.swizzle));
    return static_cast<size_t>(h % kMapSlots);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

}  // namespace

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int v = g_sms[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return 0;
    }
    g_sms[dev].store(v, std::memory_order_relaxed);
    return v;
}

cudaError_t ensure_dynamic_smem(const void *kernel, int bytes) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    cudaError_t e = cudaSuccess;
    g_optins.ensure(dev, kernel, bytes, [&] {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        return e == cudaSuccess;
    });
    return e;
}

int resident_blocks_per_sm(const void *kernel, int threads, size_t smem) {
    const int dev = current_device();
    if (dev < 0) return 0;
    return g_occ.get(
        dev, OccKey{kernel, threads, smem},
        [&] {
            int blocks = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, smem) != cudaSuccess) {
                cudaGetLastError();
                return 0;
            }
            return blocks;
        },
        [](int blocks) { return blocks > 0; });
}

int max_active_clusters(const void *kernel, int threads, size_t smem, int cluster) {
    const int dev = current_device();
    if (dev < 0) return 0;
    return g_clusters.get(
        dev, ClusterKey{kernel, threads, smem, cluster},
        [&] {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(cluster));
            cfg.blockDim = dim3(static_cast<unsigned>(threads));
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
                cudaGetLastError();
                return 0;
            }
            return n;
        },
        [](int n) { return n > 0; });
}

bool tensor_map_2d(CUtensorMap *map, const void *ptr, CUtensorMapDataType dtype, int elem_bytes,
                   int64_t rows, int64_t cols, int box_cols, int box_rows,
                   CUtensorMapSwizzle swizzle) {
    const MapKey key{ptr, rows, cols, static_cast<int>(dtype), elem_bytes, box_cols, box_rows,
                     static_cast<int>(swizzle)};
    const size_t slot = slot_of(key);
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        if (g_maps[slot].used && g_maps[slot].key == key) {
            memcpy(map, &g_maps[slot].map, sizeof(CUtensorMap));
            ++g_map_hits;
            return true;
        }
    }
    auto encode = encode_fn();
    if (!encode) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * static_cast<cuuint64_t>(elem_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMap m;
    if (encode(&m, dtype, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(g_map_mu);
    g_maps[slot].used = true;
    g_maps[slot].key = key;
    memcpy(&g_maps[slot].map, &m, sizeof(CUtensorMap));
    ++g_map_misses;
    memcpy(map, &m, sizeof(CUtensorMap));
    return true;
}

MapCacheStats map_cache_stats() {
    std::lock_guard<std::mutex> lock(g_map_mu);
    return MapCacheStats{g_map_hits, g_map_misses};
}

}  // namespace ck
