// gemv.cu -- small-M (M <= 8) ConvRot GEMV over the GEMV-resident layout, and
// the relayout that builds that layout.
//
// comfy-kitchen PR #248, "Performance improvements for qwen 3.x (Part 2)",
// Description: for M < 8 the linear is memory-bandwidth bound; interleaving
// the weights with their scales linearizes the weight stream, relayout
// kernels build that layout once, and tensor cores (not dp4a) do the math.
//
// Layout (per 16-row tile t, rows padded with zero codes / zero scales):
// K/32 blocks of 512 bytes, then the tile's 16 f32 scales.  In a block, lane l
// owns bytes [16 l, 16 l + 16): the int8 codes of the A fragments of two
// mma.m16n8k16 instructions (columns 0-15, then 16-31), in fragment-register
// order.  One coalesced 16-byte load per lane feeds two MMAs.
//
// Engine: on sm_103a the legacy INT8 mma.sync runs at ~158 TOPS, the f16 one
// at ~600 TFLOP/s, so the codes are widened to fp16 in registers (a byte
// permute onto 1024 + 128 + q and one packed subtract -- exact) and multiplied
// with mma.sync m16n8k16 into f32.  At most 32 MMAs (512 products per output,
// |sum| < 2^23) accumulate in f32 before being drained into int32, so the
// int32 result is exact.  Activation codes (fp16-held) come from the quantizer
// kernel launched just before (programmatic dependent launch: the first
// weight loads are issued before waiting on it).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ck {
namespace {

constexpr int kGemvWarps = 8;   // warps per tile (split K)
constexpr int kGemvBatch = 8;   // 512-byte blocks a lane keeps in flight per batch

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Four int8 codes -> two half2 registers holding the same integers.
// x = w ^ 0x80808080 biases each code to q + 128 in [0, 255]; placing it under
// the exponent byte 0x64 gives the fp16 value 1024 + q + 128; subtracting 1152
// leaves q exactly.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t x = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(x), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(x), "r"(0x64646464u));
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    lo = *reinterpret_cast<uint32_t *>(&ha);
    hi = *reinterpret_cast<uint32_t *>(&hb);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ldg_u32(const __half *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}

__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_packed_kernel(const __half *__restrict__ xq16, const float *__restrict__ sx, int M, int K,
                   const uint8_t *__restrict__ Wp, int N, const __nv_bfloat16 *__restrict__ bias,
                   __nv_bfloat16 *__restrict__ y) {
    __shared__ int red[kGemvWarps][32][4];
    const int tile = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int grp = lane >> 2, tg = lane & 3;
    const int nblk = K >> 5;
    const size_t tile_bytes = static_cast<size_t>(nblk) * 512 + 64;
    const uint8_t *tp = Wp + static_cast<size_t>(tile) * tile_bytes + lane * 16;
    const int per = (nblk + kGemvWarps - 1) / kGemvWarps;
    const int b_begin = min(nblk, warp * per);
    const int b_end = min(nblk, b_begin + per);
    const bool tok_ok = grp < M;
    const __half *xrow = xq16 + static_cast<size_t>(tok_ok ? grp : 0) * K + 2 * tg;

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int iacc[4] = {0, 0, 0, 0};
    int since_drain = 0;

    uint4 w[kGemvBatch];
#pragma unroll
    for (int u = 0; u < kGemvBatch; ++u)
        if (b_begin + u < b_end) w[u] = ld_stream16(tp + static_cast<size_t>(b_begin + u) * 512);
    pdl_wait();  // the activation codes come from the quantizer kernel

    for (int b = b_begin; b < b_end; b += kGemvBatch) {
        uint4 wn[kGemvBatch];
        const int bn = b + kGemvBatch;
#pragma unroll
        for (int u = 0; u < kGemvBatch; ++u)
            if (bn + u < b_end) wn[u] = ld_stream16(tp + static_cast<size_t>(bn + u) * 512);
#pragma unroll
        for (int u = 0; u < kGemvBatch; ++u) {
            if (b + u < b_end) {
                const int kb = (b + u) * 32;
                uint32_t xb0 = 0, xb1 = 0, xb2 = 0, xb3 = 0;
                if (tok_ok) {
                    xb0 = ldg_u32(xrow + kb);
                    xb1 = ldg_u32(xrow + kb + 8);
                    xb2 = ldg_u32(xrow + kb + 16);
                    xb3 = ldg_u32(xrow + kb + 24);
                }
                uint32_t a0, a1, a2, a3;
                widen4(w[u].x, a0, a1);
                widen4(w[u].y, a2, a3);
                mma16816(acc, a0, a1, a2, a3, xb0, xb1);
                widen4(w[u].z, a0, a1);
                widen4(w[u].w, a2, a3);
                mma16816(acc, a0, a1, a2, a3, xb2, xb3);
                since_drain += 2;
                if (since_drain >= 32) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        iacc[i] += __float2int_rn(acc[i]);
                        acc[i] = 0.f;
                    }
                    since_drain = 0;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kGemvBatch; ++u) w[u] = wn[u];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        iacc[i] += __float2int_rn(acc[i]);
        red[warp][lane][i] = iacc[i];
    }
    __syncthreads();
    if (warp != 0) return;
    const float *swp = reinterpret_cast<const float *>(Wp + static_cast<size_t>(tile) * tile_bytes +
                                                       static_cast<size_t>(nblk) * 512);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int tot = 0;
#pragma unroll
        for (int v = 0; v < kGemvWarps; ++v) tot += red[v][lane][i];
        // accumulator fragment: c0 (row grp, token 2tg), c1 (row grp, token 2tg+1),
        // c2 / c3 the same tokens for row grp + 8
        const int row = grp + (i >= 2 ? 8 : 0);
        const int tok = 2 * tg + (i & 1);
        const int n = tile * 16 + row;
        if (tok < M && n < N) {
            const float b = bias != nullptr ? __bfloat162float(bias[n]) : 0.0f;
            const float v = __fmaf_rn(static_cast<float>(tot) * sx[tok], swp[row], b);
            y[static_cast<size_t>(tok) * N + n] = __float2bfloat16_rn(v);
        }
    }
}

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
        const int e = j & 7;
        const int row = grp + ((e == 2 || e == 3 || e == 6 || e == 7) ? 8 : 0);
        const int col = 32 * b + 16 * (j >> 3) + 2 * tg + (j & 1) + (e >= 4 ? 8 : 0);
        const int64_t n = 16 * t + row;
        const uint32_t code = n < N ? static_cast<uint8_t>(Wq[n * K + col]) : 0u;
        word[j >> 2] |= code << (8 * (j & 3));
    }
    *reinterpret_cast<uint4 *>(out + t * tile_bytes + static_cast<size_t>(b) * 512 + lane * 16) =
        make_uint4(word[0], word[1], word[2], word[3]);
    if (b == 0 && lane < 16) {
        const int64_t n = 16 * t + lane;
        reinterpret_cast<float *>(out + t * tile_bytes + static_cast<size_t>(nblk) * 512)[lane] =
            n < N ? sw[n] : 0.0f;
    }
}

}  // namespace

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

cudaError_t launch_gemv_packed(const void *xq16, const float *sx, int64_t M, int64_t K,
                               const void *Wpacked, int64_t N, const void *bias, void *y,
                               const LaunchCtx &ctx) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + 15) / 16));
    cfg.blockDim = dim3(kGemvWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ctx.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_packed_kernel, static_cast<const __half *>(xq16), sx,
                              static_cast<int>(M), static_cast<int>(K),
                              static_cast<const uint8_t *>(Wpacked), static_cast<int>(N),
                              static_cast<const __nv_bfloat16 *>(bias),
                              static_cast<__nv_bfloat16 *>(y));
}

}  // namespace ck
