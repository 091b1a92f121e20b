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

// Register-only loop of independent mma.sync m16n8k32 s8 instructions.  The
// result is stored only if it equals a value it never takes, which keeps the
// work alive without a per-thread output buffer (sink: one int).
constexpr int kMmaIters = 1024;
constexpr int kMmaChains = 8;
__global__ void int8_mma_rate_kernel(int *sink, int seed) {
    uint32_t a0 = seed, a1 = seed + 1, a2 = seed + 2, a3 = seed + 3, b0 = seed * 3, b1 = seed * 5;
    int c[kMmaChains][4] = {};
    for (int it = 0; it < kMmaIters; ++it) {
#pragma unroll
        for (int j = 0; j < kMmaChains; ++j)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                "{%8,%9}, {%0,%1,%2,%3};"
                : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < kMmaChains; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    if (s == 0x7fffffff) *sink = s;
}

}  // namespace

cudaError_t measure_int8_mma_tops(double *tops, int *sink, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int blocks = sms * 8, threads = 256;
    cudaError_t e = cudaSuccess;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    float best_ms = 1e30f;
    for (int rep = 0; rep < 3; ++rep) {
        cudaEventRecord(e0, stream);
        int8_mma_rate_kernel<<<blocks, threads, 0, stream>>>(sink, rep + 1);
        cudaEventRecord(e1, stream);
        cudaEventSynchronize(e1);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        if (rep > 0 && ms < best_ms) best_ms = ms;
    }
    e = cudaGetLastError();
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaStreamSynchronize(stream);
    const double ops = 2.0 * 16 * 8 * 32 * kMmaChains * static_cast<double>(kMmaIters) *
                       (static_cast<double>(blocks) * threads / 32.0);
    *tops = ops / (best_ms * 1e-3) / 1e12;
    return e;
}

cudaError_t launch_stalled_wait(const LaunchCtx &ctx) {
    stalled_wait_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status,
                                                  static_cast<unsigned long long>(ctx.timeout_ns));
    return cudaGetLastError();
}

}  // namespace ck
