// gemv_fused_w6.cu -- the fused-quantizer small-M GEMV on 6-bit weight codes
// (W6A8; gemv_fused.cuh).
#include "gemv_fused.cuh"

namespace ck {

cudaError_t launch_gemv_fused_w6(const void *x, int64_t ldx, Act act, int g, int64_t M, int64_t K,
                                 const void *Wpacked, int64_t N, const void *bias,
                                 const void *residual, void *y, const LaunchCtx &ctx) {
    return gvf::launch_fused<6>(x, ldx, act, g, M, K, Wpacked, N, bias, residual, y, ctx);
}

}  // namespace ck
