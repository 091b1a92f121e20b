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
// (g = l / 4, c = l % 4) owns bytes [16 l, 16 l + 16): the A fragment of one
// mma.m16n8k32 (s8) in register order a0..a3, i.e. rows g, g + 8, g, g + 8 of
// the block by columns 8c .. 8c+3 (a0, a1) and 8c+4 .. 8c+7 (a2, a3).  The
// fragment's k index 4c + i (a0, a1) / 16 + 4c + i (a2, a3) is relabelled to
// column 8c + i / 8c + 4 + i; the activation operand gets the same relabelling,
// so the sum is unchanged and each lane reads its eight activation codes of a
// block with one 8-byte load.
//
// Engine: mma.sync m16n8k32 s8 x s8 -> s32 on the raw codes (exact for any K,
// no widening, no drains); the activation codes are the quantizer's INT8
// output.  For one or two tokens most of the MMA's eight columns would be
// padding (and GB300's INT8 MMA is slow, ~60 SM-sub-partition cycles each):
// four dp4a per token, lane and block (rows g and g + 8) do the sums instead.
//
// Streaming: two CTAs of 16 warps per SM, each walking a contiguous range of
// tiles.  Warp w owns the K-slice [w B/16, (w+1) B/16) of every tile (B = K/32
// blocks) and reads it in steps of up to 8 blocks, one 16-byte load per lane
// and block straight into registers (8 loads in flight per lane: ~128 KB of
// weights in flight per SM, the depth at which plain loads stream a 50 MB
// weight at ~5 TB/s on GB300).  The CTA's activation fragments (8 bytes per
// lane and block) are staged once in shared memory (K <= 12288; longer rows
// read them through L1).  A warp adds its tile partials into shared memory
// with integer atomics; the warp that completes a tile dequantizes it, with
// operands prefetched into shared memory at the start.  No wait in the kernel
// depends on another warp.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ck {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kStep = 8;                 // blocks per load step (8 x 16-byte loads per lane)
constexpr int kTileSlots = 32;           // most tiles one CTA handles
constexpr int kXsMaxK = 12288;           // activation fragments staged in shared memory up to here

// shared memory of one CTA handling at most tpc tiles (partials, arrival
// counts, dequantization operands), then the staged activation fragments
__host__ __device__ constexpr size_t fixed_smem(int tpc) {
    return sizeof(int) * static_cast<size_t>(tpc) * (128 + 1) + sizeof(float) * (2 * static_cast<size_t>(tpc) * 16 + 8);
}

__device__ __forceinline__ void mma_s8_16832(int (&d)[4], const uint4 &a, uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// MT (1 or 2): up to MT tokens with four dp4a per token and block (rows g and
// g + 8), summed over the lane's quad at the tile's end; MT = 8 runs the INT8
// MMA.
template <bool XS, int MT>
__global__ void __launch_bounds__(kThreads, 2)
gemv_packed_kernel(const int8_t *__restrict__ xq, const float *__restrict__ sx, int M, int K,
                   const uint8_t *__restrict__ Wp, int N, const __nv_bfloat16 *__restrict__ bias,
                   const __nv_bfloat16 *residual, __nv_bfloat16 *y, int tpc) {
    extern __shared__ __align__(16) uint8_t smem[];
    int *red = reinterpret_cast<int *>(smem);             // [tile slot][lane][4]
    int *cnt = red + tpc * 128;                           // [tile slot] warps arrived
    float *ep_sw = reinterpret_cast<float *>(cnt + tpc);  // [tile slot][16] row scales
    float *ep_b = ep_sw + tpc * 16;                       // [tile slot][16] bias
    float *ep_sx = ep_b + tpc * 16;                       // [8] token scales
    uint2 *xs = reinterpret_cast<uint2 *>(smem + (fixed_smem(tpc) + 15) / 16 * 16);  // [block][lane]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles = (N + 15) >> 4;
    const int nblk = K >> 5;
    const size_t tile_bytes = static_cast<size_t>(nblk) * 512 + 64;
    const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * tiles / gridDim.x);
    const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * tiles / gridDim.x);
    const int nslice = min(kWarps, nblk);  // warps with a K-slice
    const int sb = warp < nslice ? warp * nblk / nslice : 0;
    const int se = warp < nslice ? (warp + 1) * nblk / nslice : 0;
    const int spt = (se - sb + kStep - 1) / kStep;  // steps per tile
    const int total = spt * (t1 - t0);              // this warp's steps
    const int grp = lane >> 2, tg4 = lane & 3;

    // step i of this warp: tile t0 + i / spt, blocks sb + 8 (i % spt) ..; this
    // lane's 16 bytes of each block, loaded into registers
    uint4 w[kStep];
    auto load_step = [&](int i) {
        const int tt = t0 + i / spt;
        const int b0 = sb + (i % spt) * kStep;
        const int nb = min(kStep, se - b0);
        const uint4 *src = reinterpret_cast<const uint4 *>(
            Wp + static_cast<size_t>(tt) * tile_bytes + static_cast<size_t>(b0) * 512 + lane * 16);
#pragma unroll
        for (int j = 0; j < kStep; ++j) w[j] = j < nb ? __ldg(src + 32 * j) : make_uint4(0u, 0u, 0u, 0u);
    };
    if (total > 0) load_step(0);  // the weights do not depend on the quantizer
    // A kernel queued behind this one may launch now: it waits for our end
    // before it touches anything we read or write.
    pdl_launch_dependents();

    for (int i = threadIdx.x; i < tpc * (128 + 1); i += kThreads) red[i] = 0;
    for (int i = threadIdx.x; i < (t1 - t0) * 16; i += kThreads) {
        const int tt = t0 + i / 16, row = i % 16, n = tt * 16 + row;
        ep_sw[i] = reinterpret_cast<const float *>(Wp + static_cast<size_t>(tt) * tile_bytes +
                                                   static_cast<size_t>(nblk) * 512)[row];
        ep_b[i] = (bias != nullptr && n < N) ? __bfloat162float(bias[n]) : 0.0f;
    }
    pdl_wait();  // activation codes and scales come from the quantizer kernel
    if (threadIdx.x < 8) ep_sx[threadIdx.x] = static_cast<int>(threadIdx.x) < M ? sx[threadIdx.x] : 0.0f;
    if constexpr (XS) {
        // fragment (block b, lane l): codes 32 b + 8 (l % 4) .. + 7 of token l / 4
        for (int i = threadIdx.x; i < nblk * 32; i += kThreads) {
            const int b = i >> 5, l = i & 31, tok = (l >> 2) < M ? (l >> 2) : 0;
            xs[i] = __ldg(reinterpret_cast<const uint2 *>(xq + static_cast<size_t>(tok) * K +
                                                          32 * b + 8 * (l & 3)));
        }
    }
    __syncthreads();

    const int8_t *xrow = xq + static_cast<size_t>(grp < M ? grp : 0) * K + 8 * tg4;
    int acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
    constexpr int kCh = MT >= 4 ? 1 : 2;  // independent dp4a chains per token and row
    int dacc[kCh][MT < 8 ? MT : 1][2] = {};  // [chain][token][row g, row g + 8]
    for (int i = 0; i < total; ++i) {
        const int tt = t0 + i / spt;
        const int si = i % spt;
        const int b0 = sb + si * kStep;
        const int nb = min(kStep, se - b0);
#pragma unroll
        for (int j = 0; j < kStep; ++j) {
            if (j < nb) {
                if constexpr (MT < 8) {
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        // token t's codes 32 b + 8 c .. + 7 (token 0 stands in past M)
                        const uint2 xf = XS ? xs[(b0 + j) * 32 + 4 * t + tg4]
                                            : __ldg(reinterpret_cast<const uint2 *>(
                                                  xq + static_cast<size_t>(t < M ? t : 0) * K +
                                                  32 * (b0 + j) + 8 * tg4));
                        int &a = dacc[j % kCh][t][0], &c = dacc[j % kCh][t][1];
                        a = __dp4a(static_cast<int>(w[j].x), static_cast<int>(xf.x), a);
                        a = __dp4a(static_cast<int>(w[j].z), static_cast<int>(xf.y), a);
                        c = __dp4a(static_cast<int>(w[j].y), static_cast<int>(xf.x), c);
                        c = __dp4a(static_cast<int>(w[j].w), static_cast<int>(xf.y), c);
                    }
                } else {
                    const uint2 xf = XS ? xs[(b0 + j) * 32 + lane]
                                        : __ldg(reinterpret_cast<const uint2 *>(xrow + 32 * (b0 + j)));
                    mma_s8_16832(acc[j & 1], w[j], xf.x, xf.y);
                }
            }
        }
        if (i + 1 < total) load_step(i + 1);
        if (si == spt - 1) {
            // this warp's share of tile tt is done: add it in, the last warp dequantizes
            const int ts = tt - t0;
            int *r = red + ts * 128 + lane * 4;
            if constexpr (MT < 8) {
                // rows g, g + 8 of token t: the quad's four column ranges summed, then
                // placed where the MMA accumulator holds them (lane 4 g + t / 2)
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    int s0 = 0, s1 = 0;
#pragma unroll
                    for (int h = 0; h < kCh; ++h) {
                        s0 += dacc[h][t][0];
                        s1 += dacc[h][t][1];
                        dacc[h][t][0] = dacc[h][t][1] = 0;
                    }
                    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
                    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
                    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
                    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
                    if (tg4 == 0) {
                        int *rt = red + ts * 128 + (4 * grp + t / 2) * 4;
                        atomicAdd(rt + (t & 1), s0);
                        atomicAdd(rt + 2 + (t & 1), s1);
                    }
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) atomicAdd(r + q, acc[0][q] + acc[1][q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[0][q] = 0;
                acc[1][q] = 0;
            }
            __threadfence_block();
            __syncwarp();
            int last = 0;
            if (lane == 0) last = atomicAdd(cnt + ts, 1) == nslice - 1 ? 1 : 0;
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence_block();
                // accumulator fragment: c0 (row grp, token 2tg4), c1 (row grp,
                // token 2tg4+1), c2 / c3 the same tokens for row grp + 8
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = grp + 8 * (q >> 1);
                    const int tok = 2 * tg4 + (q & 1);
                    const int n = tt * 16 + row;
                    const int tot = *reinterpret_cast<volatile int *>(r + q);
                    if (tok < M && n < N) {
                        float v = __fmaf_rn(static_cast<float>(tot) * ep_sx[tok],
                                            ep_sw[ts * 16 + row], ep_b[ts * 16 + row]);
                        // the residual may be y itself: read before the store
                        if (residual != nullptr)
                            v += __bfloat162float(residual[static_cast<size_t>(tok) * N + n]);
                        y[static_cast<size_t>(tok) * N + n] = __float2bfloat16_rn(v);
                    }
                }
            }
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

cudaError_t launch_gemv_packed(const int8_t *xq, const float *sx, int64_t M, int64_t K,
                               const void *Wpacked, int64_t N, const void *bias,
                               const void *residual, void *y, const LaunchCtx &ctx) {
    constexpr size_t kSmemCap = 220 * 1024;  // leaves L1 to the activation fragments' loads
    const bool xs = K <= kXsMaxK;
    const size_t xs_bytes = xs ? static_cast<size_t>(K) * 8 : 0;
    static bool attr_set = false;
    if (!attr_set) {
        for (auto k : {gemv_packed_kernel<true, 1>, gemv_packed_kernel<false, 1>,
                       gemv_packed_kernel<true, 2>, gemv_packed_kernel<false, 2>,
                       gemv_packed_kernel<true, 8>, gemv_packed_kernel<false, 8>}) {
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kSmemCap));
            if (e != cudaSuccess) return e;
        }
        attr_set = true;
    }
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // two CTAs per SM when they fit, at most kTileSlots tiles each
    const int64_t tiles = (N + 15) / 16;
    int64_t grid = 0, tpc = 0;
    size_t smem = 0;
    for (int per_sm = 2; per_sm >= 1; --per_sm) {
        grid = tiles < per_sm * sms ? tiles : per_sm * sms;
        if ((tiles + grid - 1) / grid > kTileSlots) grid = (tiles + kTileSlots - 1) / kTileSlots;
        tpc = (tiles + grid - 1) / grid;
        smem = (fixed_smem(static_cast<int>(tpc)) + 15) / 16 * 16 + xs_bytes;
        if (per_sm * smem <= kSmemCap) break;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ctx.pdl ? 1 : 0;
    // dp4a for one or two tokens; from three on the INT8 MMA (measured on GB300:
    // equal at four tokens, ahead beyond)
    auto kern = M == 1   ? (xs ? gemv_packed_kernel<true, 1> : gemv_packed_kernel<false, 1>)
                : M == 2 ? (xs ? gemv_packed_kernel<true, 2> : gemv_packed_kernel<false, 2>)
                         : (xs ? gemv_packed_kernel<true, 8> : gemv_packed_kernel<false, 8>);
    return cudaLaunchKernelEx(&cfg, kern, xq,
                              sx, static_cast<int>(M), static_cast<int>(K),
                              static_cast<const uint8_t *>(Wpacked), static_cast<int>(N),
                              static_cast<const __nv_bfloat16 *>(bias),
                              static_cast<const __nv_bfloat16 *>(residual),
                              static_cast<__nv_bfloat16 *>(y), static_cast<int>(tpc));
}

}  // namespace ck
