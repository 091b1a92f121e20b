// gemv_fused.cu -- the fused-quantizer small-M GEMV on INT8 weight codes, and
// the dispatch over the weight code widths (gemv_fused.cuh).
#include "gemv_fused.cuh"

namespace ck {

bool gemv_fusable(int64_t M, int64_t K) { return gv::fusable(M, K); }

cudaError_t launch_gemv_fused_w8(const void *x, int64_t ldx, Act act, int g, int64_t M, int64_t K,
                                 const void *Wpacked, int64_t N, const void *bias,
                                 const void *residual, void *y, const LaunchCtx &ctx) {
    return gvf::launch_fused<8>(x, ldx, act, g, M, K, Wpacked, N, bias, residual, y, ctx);
}

cudaError_t launch_gemv_fused(const void *x, int64_t ldx, Act act, int g, int64_t M, int64_t K,
                              const void *Wpacked, int wbits, int64_t N, const void *bias,
                              const void *residual, void *y, const LaunchCtx &ctx) {
    switch (wbits) {
        case 8: return launch_gemv_fused_w8(x, ldx, act, g, M, K, Wpacked, N, bias, residual, y, ctx);
        case 6: return launch_gemv_fused_w6(x, ldx, act, g, M, K, Wpacked, N, bias, residual, y, ctx);
        case 4: return launch_gemv_fused_w4(x, ldx, act, g, M, K, Wpacked, N, bias, residual, y, ctx);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ck
