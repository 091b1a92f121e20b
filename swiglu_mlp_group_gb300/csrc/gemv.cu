// gemv.cu -- the relayout that builds the GEMV-resident weight layout, and the
// small-M GEMV launch on activation codes from the quantizer kernel (the
// kernel and the layout are described in gemv_kernel.cuh).
//
// comfy-kitchen PR #248, "Performance improvements for qwen 3.x (Part 2)",
// Description: relayout kernels build the interleaved weight layout once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemv_kernel.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"

namespace ck {
namespace {

using namespace gv;


// One thread per (tile, block, lane): gathers the lane's 16 codes.
__global__ void pack_gemv_kernel(const int8_t *__restrict__ Wq, const float *__restrict__ sw,
                                 int N, int K, uint8_t *__restrict__ out, int64_t total) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int nblk = K >> 5;
    const int lane = static_cast<int>(idx & 31);
    const int b = static_cast<int>((idx >> 5) % nblk);
    const int64_t t = (idx >> 5) / nblk;
    const int grp = lane >> 2, tg = lane & 3;
    const size_t tile_bytes = static_cast<size_t>(nblk) * 512 + 64;
    uint32_t word[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int reg = j >> 2;  // a0..a3
        const int row = grp + ((reg & 1) ? 8 : 0);
        const int col = 32 * b + 8 * tg + (j & 3) + ((reg & 2) ? 4 : 0);
        const int64_t n = 16 * t + row;
        const uint32_t code = n < N ? static_cast<uint8_t>(Wq[n * K + col]) : 0u;
        word[reg] |= code << (8 * (j & 3));
    }
    *reinterpret_cast<uint4 *>(out + t * tile_bytes + static_cast<size_t>(b) * 512 + lane * 16) =
        make_uint4(word[0], word[1], word[2], word[3]);
    if (b == 0 && lane < 16) {
        const int64_t n = 16 * t + lane;
        reinterpret_cast<float *>(out + t * tile_bytes + static_cast<size_t>(nblk) * 512)[lane] =
            n < N ? sw[n] : 0.0f;
    }
}

// One thread per (tile, block, lane): the lane's 16 codes as b-bit fields
// (b = 4: 8 bytes, b = 6: 12 bytes; the positions are those of the INT8
// layout, the fields as stated in include/ck.h), then the tile's scales.
__global__ void pack_gemv_lowbit_kernel(const int8_t *__restrict__ Wq, const float *__restrict__ sw,
                                        int N, int K, int bits, uint8_t *__restrict__ out,
                                        int64_t total) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int nblk = K >> 5;
    const int lane = static_cast<int>(idx & 31);
    const int b = static_cast<int>((idx >> 5) % nblk);
    const int64_t t = (idx >> 5) / nblk;
    const int grp = lane >> 2, tg = lane & 3;
    const size_t block_bytes = static_cast<size_t>(64) * bits;
    const size_t tile_bytes = static_cast<size_t>(nblk) * block_bytes + 64;
    const uint32_t mask = (1u << bits) - 1u;
    uint32_t u[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int reg = j >> 2;  // a0..a3
        const int row = grp + ((reg & 1) ? 8 : 0);
        const int col = 32 * b + 8 * tg + (j & 3) + ((reg & 2) ? 4 : 0);
        const int64_t n = 16 * t + row;
        u[j] = (n < N ? static_cast<uint32_t>(static_cast<uint8_t>(Wq[n * K + col])) : 0u) & mask;
    }
    // the lane's words 0 and 1 at 8 lane, word 2 (6-bit) at 256 + 4 lane
    uint8_t *lp = out + t * tile_bytes + static_cast<size_t>(b) * block_bytes + 8 * lane;
    if (bits == 4) {
        // word 0: a0 in the low nibbles, a1 in the high ones; word 1: a2, a3
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            w[h] = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) w[h] |= (u[8 * h + i] | u[8 * h + 4 + i] << 4) << (8 * i);
        }
        *reinterpret_cast<uint2 *>(lp) = make_uint2(w[0], w[1]);
    } else {
        // words 0..2: a0..a2 in bits 2..7 of each byte, a3 split into 2-bit
        // pieces in bits 0..1 (low piece in word 0)
        uint32_t w[3];
#pragma unroll
        for (int wi = 0; wi < 3; ++wi) {
            w[wi] = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[wi] |= ((u[4 * wi + i] << 2) | ((u[12 + i] >> (2 * wi)) & 3u)) << (8 * i);
        }
        *reinterpret_cast<uint2 *>(lp) = make_uint2(w[0], w[1]);
        *reinterpret_cast<uint32_t *>(lp + 256 - 4 * lane) = w[2];
    }
    if (b == 0 && lane < 16) {
        const int64_t n = 16 * t + lane;
        reinterpret_cast<float *>(out + t * tile_bytes + static_cast<size_t>(nblk) * block_bytes)[lane] =
            n < N ? sw[n] : 0.0f;
    }
}

}  // namespace

size_t gemv_packed_lowbit_bytes(int64_t N, int64_t K, int bits) {
    const int64_t tiles = (N + 15) / 16;
    return static_cast<size_t>(tiles) * (static_cast<size_t>(K) / 32 * 64 * bits + 64);
}

cudaError_t launch_pack_gemv_lowbit(const int8_t *Wq, const float *sw, int64_t N, int64_t K,
                                    int bits, void *out, cudaStream_t stream) {
    if (bits != 4 && bits != 6) return cudaErrorInvalidValue;
    const int64_t total = (N + 15) / 16 * (K / 32) * 32;
    const int threads = 256;
    pack_gemv_lowbit_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0,
                              stream>>>(Wq, sw, static_cast<int>(N), static_cast<int>(K), bits,
                                        static_cast<uint8_t *>(out), total);
    return cudaGetLastError();
}

size_t gemv_packed_bytes(int64_t N, int64_t K) {
    const int64_t tiles = (N + 15) / 16;
    return static_cast<size_t>(tiles) * (static_cast<size_t>(K) * 16 + 64);
}

cudaError_t launch_pack_gemv(const int8_t *Wq, const float *sw, int64_t N, int64_t K, void *out,
                             cudaStream_t stream) {
    const int64_t total = (N + 15) / 16 * (K / 32) * 32;
    const int threads = 256;
    pack_gemv_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, stream>>>(
        Wq, sw, static_cast<int>(N), static_cast<int>(K), static_cast<uint8_t *>(out), total);
    return cudaGetLastError();
}

namespace {

template <int WB, bool S32>
cudaError_t launch_packed_wb(const int8_t *xq, const float *sx, int64_t M, int64_t K,
                             const void *Wpacked, int64_t N, const void *bias,
                             const void *residual, void *y, const LaunchCtx &ctx) {
    const bool xs = stage_xs(M, K, false, WB);
    // the shared-memory opt-in belongs to each device's copy of a kernel
    for (auto k : {gemv_packed_kernel<true, 1, -1, 0, WB, S32>, gemv_packed_kernel<false, 1, -1, 0, WB, S32>,
                   gemv_packed_kernel<true, 2, -1, 0, WB, S32>, gemv_packed_kernel<false, 2, -1, 0, WB, S32>,
                   gemv_packed_kernel<true, 8, -1, 0, WB, S32>, gemv_packed_kernel<false, 8, -1, 0, WB, S32>}) {
        cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(k), static_cast<int>(kSmemCap));
        if (e != cudaSuccess) return e;
    }
    const int sms = sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
    const Plan p = plan(M, K, N, sms, false, WB);
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
    // dp4a for few tokens, the INT8 MMA beyond (engine_tokens)
    const int mt = engine_tokens(M, false, WB);
    if constexpr (WB == 8) {
        for (auto k : {gemv_packed_kernel<true, 4, -1, 0, 8, S32>, gemv_packed_kernel<false, 4, -1, 0, 8, S32>}) {
            cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(k), static_cast<int>(kSmemCap));
            if (e != cudaSuccess) return e;
        }
    }
    auto kern = mt == 1   ? (xs ? gemv_packed_kernel<true, 1, -1, 0, WB, S32> : gemv_packed_kernel<false, 1, -1, 0, WB, S32>)
                : mt == 2 ? (xs ? gemv_packed_kernel<true, 2, -1, 0, WB, S32> : gemv_packed_kernel<false, 2, -1, 0, WB, S32>)
                          : (xs ? gemv_packed_kernel<true, 8, -1, 0, WB, S32> : gemv_packed_kernel<false, 8, -1, 0, WB, S32>);
    if constexpr (WB == 8) {
        if (mt == 4)
            kern = xs ? gemv_packed_kernel<true, 4, -1, 0, WB, S32> : gemv_packed_kernel<false, 4, -1, 0, WB, S32>;
    }
    // The weights may be read before the wait: launched behind this library's
    // quantizer they are settled by the time it lets this kernel in, launched
    // alone without the programmatic attribute nothing is ahead of it, and
    // launched alone with it the caller declared them settled.
    return cudaLaunchKernelEx(&cfg, kern, xq, sx, static_cast<const __nv_bfloat16 *>(nullptr),
                              static_cast<int64_t>(0), static_cast<int>(M), static_cast<int>(K),
                              static_cast<const uint8_t *>(Wpacked), static_cast<int>(N),
                              static_cast<const __nv_bfloat16 *>(bias),
                              static_cast<const __nv_bfloat16 *>(residual),
                              static_cast<__nv_bfloat16 *>(y), static_cast<int>(p.tpc), 1);
}

}  // namespace

cudaError_t launch_gemv_packed(const int8_t *xq, const float *sx, int64_t M, int64_t K,
                               const void *Wpacked, int wbits, int64_t N, const void *bias,
                               const void *residual, void *y, const LaunchCtx &ctx,
                               int32_t *acc_out) {
    if (acc_out != nullptr) {
        switch (wbits) {
            case 8: return launch_packed_wb<8, true>(xq, sx, M, K, Wpacked, N, nullptr, nullptr, acc_out, ctx);
            case 6: return launch_packed_wb<6, true>(xq, sx, M, K, Wpacked, N, nullptr, nullptr, acc_out, ctx);
            case 4: return launch_packed_wb<4, true>(xq, sx, M, K, Wpacked, N, nullptr, nullptr, acc_out, ctx);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (wbits) {
        case 8: return launch_packed_wb<8, false>(xq, sx, M, K, Wpacked, N, bias, residual, y, ctx);
        case 6: return launch_packed_wb<6, false>(xq, sx, M, K, Wpacked, N, bias, residual, y, ctx);
        case 4: return launch_packed_wb<4, false>(xq, sx, M, K, Wpacked, N, bias, residual, y, ctx);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ck
