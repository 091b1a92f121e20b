// launch_util.h -- host-side launch bookkeeping shared by the kernels'
// launchers: per-device facts looked up once, the per-(device, kernel)
// shared-memory opt-in, and a cache of TMA tensor maps.  All of it is
// thread-safe; nothing here allocates device memory.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ck {

// Index of the current CUDA device, or -1.
int current_device();

// SM count of the current device (looked up once per device; 0 on error).
int sm_count();

// Opts `kernel` into `bytes` of dynamic shared memory on the current device,
// once per (device, kernel): the attribute belongs to each device's copy of
// the kernel, so a second device in the process needs its own call.
cudaError_t ensure_dynamic_smem(const void *kernel, int bytes);

// Thread blocks of `kernel` resident per SM on the current device with
// `threads` threads and `smem` bytes of dynamic shared memory (cached per
// (device, kernel, threads, smem)); 0 on error.
int resident_blocks_per_sm(const void *kernel, int threads, size_t smem);

// Clusters of `cluster` blocks of `kernel` (x-dimension clusters, `threads`
// threads, `smem` bytes of dynamic shared memory each) that the current device
// holds at once (cached per (device, kernel, threads, smem, cluster)); 0 on
// error.  The kernel's shared-memory opt-in must be done first.
int max_active_clusters(const void *kernel, int threads, size_t smem, int cluster);

// A 2-D row-major tensor map: `rows` rows of `cols` elements of `elem_bytes`
// bytes, row stride cols * elem_bytes, box of box_cols x box_rows, out-of-range
// elements read as zero.  Maps are cached by value (pointer, type, shape, box,
// swizzle): the same request returns the same bytes without re-encoding them.
bool tensor_map_2d(CUtensorMap *map, const void *ptr, CUtensorMapDataType dtype, int elem_bytes,
                   int64_t rows, int64_t cols, int box_cols, int box_rows,
                   CUtensorMapSwizzle swizzle);

// Host-side counters of the map cache (tests and the bench read them).
struct MapCacheStats {
    uint64_t hits, misses;
};
MapCacheStats map_cache_stats();

}  // namespace ck
