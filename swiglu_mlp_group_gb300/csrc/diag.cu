// diag.cu -- test hook for the bounded-wait machinery (a kernel whose barrier
// is never completed, so its wait runs out, records the timeout in the device
// status word and returns; nothing in it can hang: the wait is bounded by the
// same time limit every pipeline wait of the library uses), and the two
// tensor-core rate diagnostics the measurements quote peaks against.
#include "internal.h"
#include "launch_util.h"
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

// try_wait on phase 0 of `bar` until it completes or `timeout_ns` passes
__device__ __forceinline__ bool mbar_wait_drain_plain(uint32_t bar, unsigned long long timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, 0))
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    return true;
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
    const int sms = sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
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

namespace {

// Back-to-back tcgen05.mma kind::f16 (M = 128, N = 256, K = 16) from shared
// memory, issued by one thread per SM into two alternating TMEM accumulators:
// the instruction's own rate, without TMA or an epilogue (zero operands).  One commit at the end; its wait
// is bounded (a timeout records kDeviceStatusTimeout, then waits again, bounded,
// before TMEM is freed).
constexpr int kUmmaIters = 2048;  // x 4 instructions
constexpr int kUmmaSmem = 120 * 1024;  // one CTA per SM
__global__ void __launch_bounds__(128, 1) tcgen05_rate_kernel(unsigned int *status,
                                                               unsigned long long timeout_ns) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t slot;
    const uint32_t raw = smem_u32(smem_raw);
    // A: 128 x 64 fp16 (16 KB); B: 256 x 64 (32 KB)
    const uint32_t base = (raw + 1023u) & ~1023u;
    for (int i = threadIdx.x; i < 49152 / 16; i += blockDim.x)
        *reinterpret_cast<uint4 *>(smem_raw + (base - raw) + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    const uint32_t bar_s = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(bar_s, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(smem_u32(&slot), 512);
        tmem_relinquish();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = slot;
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc = idesc_f16_f32(128, 256);
        const uint64_t ad = sdesc_kmajor_sw128(base), bd = sdesc_kmajor_sw128(base + 16384);
        for (int it = 0; it < kUmmaIters; ++it) {
            const uint32_t d = tmem + static_cast<uint32_t>((it & 1) * 256);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_f16_ss(d, ad + 2u * k, bd + 2u * k, idesc, (it > 1 || k > 0) ? 1u : 0u);
        }
        mma_commit(bar_s);
    }
    if (threadIdx.x == 0) {
        if (!mbar_wait_drain_plain(bar_s, timeout_ns)) {
            atomicOr(status, kDeviceStatusTimeout);
            mbar_wait_drain_plain(bar_s, timeout_ns);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t measure_tcgen05_f16_tflops(double *tflops, const LaunchCtx &ctx) {
    const int sms = sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(tcgen05_rate_kernel), kUmmaSmem);
    if (e != cudaSuccess) return e;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    float best_ms = 1e30f;
    for (int rep = 0; rep < 3 && e == cudaSuccess; ++rep) {
        cudaEventRecord(e0, ctx.stream);
        tcgen05_rate_kernel<<<sms, 128, kUmmaSmem, ctx.stream>>>(
            ctx.status, static_cast<unsigned long long>(ctx.timeout_ns));
        e = cudaGetLastError();
        cudaEventRecord(e1, ctx.stream);
        cudaEventSynchronize(e1);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        if (rep > 0 && ms < best_ms) best_ms = ms;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaStreamSynchronize(ctx.stream);
    if (e != cudaSuccess) return e;
    const double flops = 2.0 * 128 * 256 * 16 * 4.0 * kUmmaIters * sms;
    *tflops = flops / (best_ms * 1e-3) / 1e12;
    return cudaSuccess;
}

cudaError_t launch_stalled_wait(const LaunchCtx &ctx) {
    stalled_wait_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status, static_cast<unsigned long long>(ctx.timeout_ns));
    return cudaGetLastError();
}

}  // namespace ck
