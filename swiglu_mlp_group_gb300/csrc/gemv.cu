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
// Streaming: a persistent grid (two CTAs per SM); in each CTA one producer
// lane streams the weight tiles with 1-D bulk copies (cp.async.bulk) through a
// 6-stage (16 KB each) shared-memory ring, and eight consumer warps read the fragments from
// shared memory.  The weights do not depend on the quantizer, so the stream
// starts before the wait on it; every wait is bounded in time.
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

#ifndef CK_GEMV_CHUNK_BLOCKS
#define CK_GEMV_CHUNK_BLOCKS 32
#endif
#ifndef CK_GEMV_STAGES
#define CK_GEMV_STAGES 6
#endif
#ifndef CK_GEMV_TILE_GROUP
#define CK_GEMV_TILE_GROUP 4
#endif
#ifndef CK_GEMV_CTAS_PER_SM
#define CK_GEMV_CTAS_PER_SM 2
#endif
constexpr int kConsumers = 8;                 // consumer warps (split each chunk's blocks)
constexpr int kThreads = 32 * (kConsumers + 1);  // + one producer warp
constexpr int kChunkBlocks = CK_GEMV_CHUNK_BLOCKS;  // 512-byte blocks per stage (16 KB)
constexpr int kStageBytes = kChunkBlocks * 512;
constexpr int kStages = CK_GEMV_STAGES;       // 96 KB of the weight stream in flight per CTA
constexpr int kTileGroup = CK_GEMV_TILE_GROUP;  // tiles sharing one load of x fragments
constexpr int kCtasPerSm = CK_GEMV_CTAS_PER_SM;
constexpr int kBlocksPerWarp = kChunkBlocks / kConsumers;
constexpr size_t kSmemBytes = static_cast<size_t>(kStages) * kStageBytes +
                              sizeof(int) * kConsumers * kTileGroup * 32 * 4 + 8 * (2 * kStages) +
                              16 + 128;

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

__device__ __forceinline__ uint4 lds_u128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Persistent GEMV.  CTA c owns the contiguous tile range
// [c * tiles / grid, (c + 1) * tiles / grid) and walks it in groups of up to
// kTileGroup tiles; for each K-chunk of 16 blocks it streams the group's tile
// chunks through the ring (warp 0, one lane, cp.async.bulk).  Consumer warp w
// handles blocks w and w + 8 of every chunk: its x fragments are loaded once
// per chunk and reused for every tile of the group.
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
gemv_packed_kernel(const __half *__restrict__ xq16, const float *__restrict__ sx, int M, int K,
                   const uint8_t *__restrict__ Wp, int N, const __nv_bfloat16 *__restrict__ bias,
                   __nv_bfloat16 *__restrict__ y, unsigned int *status,
                   unsigned long long timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = (128u - (raw_s & 127u)) & 127u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t ring_s = raw_s + pad;
    int *red = reinterpret_cast<int *>(smem + kStages * kStageBytes);  // [w][tg][lane][4]
    const uint32_t bars_s =
        ring_s + kStages * kStageBytes + sizeof(int) * kConsumers * kTileGroup * 32 * 4;
    auto full_bar = [&](int st) { return bars_s + 8u * st; };
    auto empty_bar = [&](int st) { return bars_s + 8u * (kStages + st); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(
        smem + kStages * kStageBytes + sizeof(int) * kConsumers * kTileGroup * 32 * 4 +
        8 * 2 * kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles = (N + 15) >> 4;
    const int nblk = K >> 5;
    const int nchunk = (nblk + kChunkBlocks - 1) / kChunkBlocks;
    const size_t tile_bytes = static_cast<size_t>(nblk) * 512 + 64;
    const int t_begin = static_cast<int>(static_cast<int64_t>(blockIdx.x) * tiles / gridDim.x);
    const int t_end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * tiles / gridDim.x);
    const WaitCtl ctl{abort_flag, status, timeout_ns};

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(full_bar(st), 1);
            mbar_init(empty_bar(st), kConsumers);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int g0 = t_begin; g0 < t_end && ok; g0 += kTileGroup) {
                const int ntg = min(kTileGroup, t_end - g0);
                for (int c = 0; c < nchunk && ok; ++c) {
                    const int nb = min(kChunkBlocks, nblk - c * kChunkBlocks);
                    for (int tg = 0; tg < ntg; ++tg) {
                        if (!mbar_wait(empty_bar(stage), ph ^ 1u, ctl)) {
                            ok = false;
                            break;
                        }
                        const uint8_t *src = Wp + static_cast<size_t>(g0 + tg) * tile_bytes +
                                             static_cast<size_t>(c) * kStageBytes;
                        mbar_arrive_expect_tx(full_bar(stage), nb * 512);
                        bulk_load_1d(ring_s + stage * kStageBytes, src, nb * 512, full_bar(stage));
                        ++issued;
                        if (++stage == kStages) {
                            stage = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
            if (!ok) {
                // let the copies still in flight land before the CTA exits
                const int first = issued > kStages ? issued - kStages : 0;
                for (int i = first; i < issued; ++i) {
                    const uint32_t bar = full_bar(i % kStages), par = (i / kStages) & 1;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(bar, par) && globaltimer_ns() - t0 < timeout_ns) {
                    }
                }
            }
        }
        return;  // the producer takes no part in the consumer barriers below
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int grp = lane >> 2, tg4 = lane & 3;
    const bool tok_ok = grp < M;
    const __half *xrow = xq16 + static_cast<size_t>(tok_ok ? grp : 0) * K + 2 * tg4;
    pdl_wait();  // x codes and scales come from the quantizer kernel
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int g0 = t_begin; g0 < t_end; g0 += kTileGroup) {
        const int ntg = min(kTileGroup, t_end - g0);
        // Warp cw < ntg dequantizes tile g0 + cw at the end of the group; its
        // scales, bias and token scales are loaded now, off the critical path.
        float ep_sw[2] = {0.f, 0.f}, ep_b[2] = {0.f, 0.f}, ep_sx[2] = {0.f, 0.f};
        if (cw < ntg) {
            const int tile = g0 + cw;
            const float *swp = reinterpret_cast<const float *>(
                Wp + static_cast<size_t>(tile) * tile_bytes + static_cast<size_t>(nblk) * 512);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int row = grp + 8 * r;
                const int n = tile * 16 + row;
                ep_sw[r] = swp[row];
                if (bias != nullptr && n < N) ep_b[r] = __bfloat162float(bias[n]);
                const int tok = 2 * tg4 + r;
                if (tok < M) ep_sx[r] = sx[tok];
            }
        }
        float acc[kTileGroup][4];
        int iacc[kTileGroup][4];
#pragma unroll
        for (int tg = 0; tg < kTileGroup; ++tg)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[tg][i] = 0.f;
                iacc[tg][i] = 0;
            }
        int since_drain = 0;
        // x fragments of this warp's blocks (cw, cw + 8) of a chunk; the next
        // chunk's are loaded one chunk ahead
        auto load_x = [&](int c, uint32_t (&xb)[kBlocksPerWarp][4]) {
#pragma unroll
            for (int h = 0; h < kBlocksPerWarp; ++h) {
                const int b = c * kChunkBlocks + cw + kConsumers * h;
                const bool has = c < nchunk && b < nblk && tok_ok;
#pragma unroll
                for (int q = 0; q < 4; ++q) xb[h][q] = has ? ldg_u32(xrow + b * 32 + 8 * q) : 0u;
            }
        };
        // Chunk c consumes x fragments loaded two chunks earlier: the loop is
        // unrolled by two over buffers xa / xb so a register filled by a load
        // is first read where it is used (no register copies that would wait
        // on the load).
        auto process_chunk = [&](int c, const uint32_t (&xf)[kBlocksPerWarp][4]) {
            bool has[kBlocksPerWarp];
#pragma unroll
            for (int h = 0; h < kBlocksPerWarp; ++h)
                has[h] = c * kChunkBlocks + cw + kConsumers * h < nblk;
#pragma unroll
            for (int tg = 0; tg < kTileGroup; ++tg) {
                if (tg < ntg && ok) {
                    int got = 0;
                    if (lane == 0) got = mbar_wait(full_bar(stage), ph, ctl) ? 1 : 0;
                    got = __shfl_sync(0xffffffffu, got, 0);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    const uint32_t sbase = ring_s + stage * kStageBytes + lane * 16;
#pragma unroll
                    for (int h = 0; h < kBlocksPerWarp; ++h) {
                        if (has[h]) {
                            const uint4 w = lds_u128(sbase + (cw + kConsumers * h) * 512);
                            uint32_t a0, a1, a2, a3;
                            widen4(w.x, a0, a1);
                            widen4(w.y, a2, a3);
                            mma16816(acc[tg], a0, a1, a2, a3, xf[h][0], xf[h][1]);
                            widen4(w.z, a0, a1);
                            widen4(w.w, a2, a3);
                            mma16816(acc[tg], a0, a1, a2, a3, xf[h][2], xf[h][3]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty_bar(stage));
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            // 2 MMAs per block per tile: drain before 512 products pile up
            since_drain += 2 * kBlocksPerWarp;
            if (since_drain >= 32) {
#pragma unroll
                for (int tg = 0; tg < kTileGroup; ++tg)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        iacc[tg][i] += __float2int_rn(acc[tg][i]);
                        acc[tg][i] = 0.f;
                    }
                since_drain = 0;
            }
        };
        uint32_t xa[kBlocksPerWarp][4], xb[kBlocksPerWarp][4];
        load_x(0, xa);
        load_x(1, xb);
        for (int c = 0; c < nchunk && ok; c += 2) {
            process_chunk(c, xa);
            load_x(c + 2, xa);
            if (c + 1 < nchunk && ok) {
                process_chunk(c + 1, xb);
                load_x(c + 3, xb);
            }
        }
#pragma unroll
        for (int tg = 0; tg < kTileGroup; ++tg)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                iacc[tg][i] += __float2int_rn(acc[tg][i]);
                red[((cw * kTileGroup + tg) * 32 + lane) * 4 + i] = iacc[tg][i];
            }
        named_bar_sync(1, kConsumers * 32);
        if (cw < ntg && ok) {
            const int tile = g0 + cw;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                int tot = 0;
#pragma unroll
                for (int v = 0; v < kConsumers; ++v)
                    tot += red[((v * kTileGroup + cw) * 32 + lane) * 4 + i];
                // accumulator fragment: c0 (row grp, token 2tg4), c1 (row grp,
                // token 2tg4+1), c2 / c3 the same tokens for row grp + 8
                const int r = i >> 1;
                const int row = grp + 8 * r;
                const int tok = 2 * tg4 + (i & 1);
                const int n = tile * 16 + row;
                if (tok < M && n < N) {
                    const float v = __fmaf_rn(static_cast<float>(tot) * ep_sx[i & 1], ep_sw[r], ep_b[r]);
                    y[static_cast<size_t>(tok) * N + n] = __float2bfloat16_rn(v);
                }
            }
        }
        // red is reused by the next group; leave together if any warp gave up
        if (named_bar_or(1, kConsumers * 32, !ok || *abort_flag != 0)) break;
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
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemv_packed_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles = (N + 15) / 16;
    const int64_t grid = tiles < kCtasPerSm * sms ? tiles : kCtasPerSm * sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
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
                              static_cast<__nv_bfloat16 *>(y), ctx.status,
                              static_cast<unsigned long long>(ctx.timeout_ns));
}

}  // namespace ck
