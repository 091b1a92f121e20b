// gemv.cu -- small-M GEMV (placeholder until the packed layout lands).
#include "internal.h"

namespace ck {

size_t gemv_packed_bytes(int64_t N, int64_t K) {
    const int64_t tiles = (N + 15) / 16;
    return static_cast<size_t>(tiles) * (static_cast<size_t>(K) * 16 + 64);
}

cudaError_t launch_pack_gemv(const int8_t *, const float *, int64_t, int64_t, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t launch_gemv_packed(const void *, const float *, int64_t, int64_t, const void *, int64_t,
                               const void *, void *, const LaunchCtx &) {
    return cudaErrorNotSupported;
}

}  // namespace ck
