// diag.cu -- test hook for the bounded-wait machinery: a kernel whose barrier
// is never completed, so its wait runs out, records the timeout in the device
// status word and returns.  Nothing in it can hang: the wait is bounded by the
// same time limit every pipeline wait of the library uses.
#include "internal.h"
#include "ptx.cuh"

namespace ck {
namespace {

__global__ void stalled_wait_kernel(unsigned int *status, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);  // expects one arrival that never comes
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtl ctl{&abort_flag, status, timeout_ns};
        mbar_wait(smem_u32(&bar), 0, ctl);
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_stalled_wait(const LaunchCtx &ctx) {
    stalled_wait_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status,
                                                  static_cast<unsigned long long>(ctx.timeout_ns));
    return cudaGetLastError();
}

}  // namespace ck
