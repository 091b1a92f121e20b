// gemv_fused.cuh -- the small-M GEMV launch whose CTAs quantize the few
// activation rows themselves: one kernel per call instead of the quantizer
// kernel plus the GEMV (the kernel is described in gemv_kernel.cuh).  One
// translation unit per weight code width instantiates it (gemv_fused.cu,
// gemv_fused_w6.cu, gemv_fused_w4.cu), so that they compile in parallel.
//
// comfy-kitchen PR #248, "Performance improvements for qwen 3.x (Part 2)",
// Description: the small-M activation is quantized per CTA into shared memory.
#pragma once

#include <cuda_bf16.h>

#include "gemv_kernel.cuh"
#include "internal.h"
#include "launch_util.h"

namespace ck {
namespace gvf {

using namespace gv;

template <int MT, int ACT, int WB>
auto pick_g(int g) {
    return g == 64    ? gemv_packed_kernel<true, MT, ACT, 64, WB>
           : g == 128 ? gemv_packed_kernel<true, MT, ACT, 128, WB>
                      : gemv_packed_kernel<true, MT, ACT, 256, WB>;
}

template <int MT, int WB>
auto pick_act(Act act, int g) {
    return act == Act::kSwiglu ? pick_g<MT, 1, WB>(g) : pick_g<MT, 0, WB>(g);
}

template <int WB>
auto pick(int64_t M, Act act, int g) {
    const int mt = engine_tokens(M, true, WB);
    auto k = mt == 1 ? pick_act<1, WB>(act, g) : mt == 2 ? pick_act<2, WB>(act, g) : pick_act<8, WB>(act, g);
    if constexpr (WB == 8) {
        if (mt == 4) k = pick_act<4, WB>(act, g);
    }
    return k;
}

template <int WB>
cudaError_t launch_fused(const void *x, int64_t ldx, Act act, int g, int64_t M, int64_t K,
                         const void *Wpacked, int64_t N, const void *bias, const void *residual,
                         void *y, const LaunchCtx &ctx) {
    if (!fusable(M, K) || M < 1 || M > 8 || K % g != 0 || (g != 64 && g != 128 && g != 256))
        return cudaErrorInvalidValue;
    // the shared-memory opt-in belongs to each device's copy of a kernel
    for (int64_t mm : {1, 2, 3, 8})
        for (Act a : {Act::kNone, Act::kSwiglu})
            for (int gg : {64, 128, 256}) {
                cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(pick<WB>(mm, a, gg)),
                                                    static_cast<int>(kSmemCap));
                if (e != cudaSuccess) return e;
            }
    const int sms = sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
    const Plan p = plan(M, K, N, sms, true, WB);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ctx.pdl ? 1 : 0;
    // x is read after the wait on the kernel ahead; the weights before it only
    // when the caller declared them settled
    return cudaLaunchKernelEx(&cfg, pick<WB>(M, act, g), static_cast<const int8_t *>(nullptr),
                              static_cast<const float *>(nullptr),
                              static_cast<const __nv_bfloat16 *>(x), ldx, static_cast<int>(M),
                              static_cast<int>(K), static_cast<const uint8_t *>(Wpacked),
                              static_cast<int>(N), static_cast<const __nv_bfloat16 *>(bias),
                              static_cast<const __nv_bfloat16 *>(residual),
                              static_cast<__nv_bfloat16 *>(y), static_cast<int>(p.tpc),
                              ctx.early_trigger ? 1 : 0);
}

}  // namespace gvf
}  // namespace ck
