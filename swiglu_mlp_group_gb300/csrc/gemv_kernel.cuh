// gemv_kernel.cuh -- the small-M (M <= 8) ConvRot GEMV kernel over the
// GEMV-resident layout, instantiated by gemv.cu (activation codes from the
// quantizer kernel) and gemv_fused.cu (each CTA quantizes the activation rows
// itself).
//
// comfy-kitchen PR #248, "Performance improvements for qwen 3.x (Part 2)",
// Description: for M < 8 the linear is memory-bandwidth bound; interleaving
// the weights with their scales linearizes the weight stream, relayout
// kernels build that layout once, the activation is quantized per CTA into
// shared memory, and the PR has tensor cores rather than dp4a do the math.
// Here the INT8 tensor-core MMA does it from three (INT8 weights: five)
// tokens on; for fewer tokens dp4a does (see Engine below: a departure from
// the PR, measured faster on GB300).  Commits and Description also name 4- and 6-bit weight
// decode: the W6A8 / W4A8 layouts (WFmt) decode to the INT8 fragments in
// registers and run the same engine.
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
// no widening, no drains).  For a few tokens most of the MMA's eight columns
// would be padding (and GB300's INT8 MMA is slow, ~60 SM-sub-partition cycles
// each): four dp4a per token, lane and block (rows g and g + 8) do the sums
// instead -- for one or two tokens, and for three or four on INT8 weights
// (engine_tokens).  An f16 tensor-core form of the MMA engine (codes widened
// to f16 in registers by a byte permute and a packed subtraction, two
// m16n8k16 per block, f32 sums exact below 2^24 and added into int32 per
// load step) measured 0.6-3.1 us slower on 6-bit and 4-bit weights and at
// 4096 x 12288, 0.6 us faster only at 18432 x 3072: the widening costs more
// issue slots than the INT8 MMA pipe it relieves.  (tcgen05 has no INT8 kind on sm_103a, and its 128-row tiles
// would be 94-97% padding at M <= 8.)
//
// Streaming: two CTAs of 16 warps per SM, each walking a contiguous range of
// tiles.  Warp w owns the K-slice [w B/16, (w+1) B/16) of every tile (B = K/32
// blocks) and reads it in steps of up to 8 blocks, one 16-byte load per lane
// and block straight into registers (8 loads in flight per lane: ~128 KB of
// weights in flight per SM, the depth at which plain loads stream a 50 MB
// weight at ~5 TB/s on GB300; the 6- and 4-bit layouts take the same 8-block
// steps of 12 and 8 bytes per lane, so 3/4 and 1/2 of those bytes in flight:
// longer steps left unrolled iterations idle at the workloads' K-slices).
// A TMA-fed variant (one producer warp streaming 8 KB stages into a
// shared-memory ring for sixteen MMA warps) ran 2.3x slower on GB300: its
// copies were issued ~330 ns apart per SM (~25 GB/s per SM), whether as 2-D
// tensor or 1-D bulk copies.  Bulk L2 prefetches of each warp's later steps,
// issued at the start, made every case 0.1-4 us slower as well.  The CTA's activation fragments (8 bytes per
// lane and block) live in shared memory (up to 48 KB of them; beyond, the
// warps read them through L1).  A warp adds its tile partials into shared
// memory with integer atomics; the warp that completes a tile dequantizes it,
// with operands prefetched into shared memory at the start.  No wait in the
// kernel depends on another warp.
//
// Fused quantization (FQ >= 0, act none / swiglu; M * round_up(K/32, 32) <=
// 512): the CTA's first M teams of round_up(K/32, 32) threads rotate and
// quantize one activation row each -- the standalone quantizer's arithmetic
// (quant_core.cuh), so the codes are the same bit for bit -- straight into the
// fragment layout, while the other warps' first weight steps are in flight
// into their registers and L2 fetches the quantizing warps' first two steps
// (bulk prefetch, no registers held), which those load once done.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_core.cuh"

namespace ck {
namespace gv {

using namespace qc;

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kTileSlots = 32;           // most tiles one CTA handles
// activation fragments staged in shared memory up to this size per CTA; larger
// ones are read through L1.  Measured on GB300 (budgets 16-96 KB): at 96 KB the
// eight-token fragments of K = 12288 (two CTAs of 97 KB) leave L1 too small for
// the weight loads in flight, 2.0 us slower than reading them through L1; at
// 16 KB the K = 4096 ones lose 0.5-1.3 us.
constexpr size_t kXsMaxBytes = 48 * 1024;
constexpr size_t kSmemCap = 220 * 1024;  // leaves L1 to the activation fragments' loads

// shared memory of one CTA handling at most tpc tiles (partials, arrival
// counts, dequantization operands, the fused quantizer's warp maxima), then
// the activation fragments.  Kept small: what shared memory does not take, L1
// keeps for the weight loads in flight (at two CTAs of ~97 KB a few hundred
// bytes more cost GB300 the next carveout step and 2.5 us at K = 12288).
__host__ __device__ constexpr size_t fixed_smem(int tpc) {
    return sizeof(int) * static_cast<size_t>(tpc) * (128 + 1) +
           sizeof(float) * (2 * static_cast<size_t>(tpc) * 16 + 8 + kWarps);
}
// The engine's token count MT for M tokens of wb-bit weights: dp4a for one
// or two tokens, and for three or four on INT8 weights in the two-kernel
// path; the MMA (8 slots) beyond.  Measured on GB300 (kernel alone, three
// weight shapes, M = 3 / 4): dp4a ahead of the MMA by 0.1-0.6 us on INT8
// weights, behind it by 0.1-1.4 us on 6-bit ones (their decode costs more
// ALU), mixed on 4-bit ones.  The activation fragments hold MT tokens.
__host__ __device__ constexpr int engine_tokens(int64_t M, bool fused, int wb) {
    return M <= 2 ? static_cast<int>(M) : (M <= 4 && wb == 8) ? 4 : 8;
}
__host__ __device__ constexpr int frag_tokens(int64_t M, bool fused, int wb) {
    return engine_tokens(M, fused, wb);
}

// Whether the CTA stages the activation fragments in shared memory (else the
// warps read them through L1).
__host__ __device__ constexpr bool stage_xs(int64_t M, int64_t K, bool fused, int wb) {
    return static_cast<size_t>(K) * frag_tokens(M, fused, wb) <= kXsMaxBytes;
}
// Whether one CTA can quantize all M rows itself (one 32-element unit per
// thread at most, the fragments staged in shared memory).
__host__ __device__ constexpr bool fusable(int64_t M, int64_t K) {
    return stage_xs(M, K, true, 8) && stage_xs(M, K, true, 6) && M * ((K / 32 + 31) / 32 * 32) <= kThreads;
}

struct Plan {
    int64_t grid, tpc;
    size_t smem;
};
// two CTAs per SM when they fit, at most kTileSlots tiles each
inline Plan plan(int64_t M, int64_t K, int64_t N, int sms, bool fused, int wb) {
    const size_t xs_bytes =
        stage_xs(M, K, fused, wb) ? static_cast<size_t>(K) * frag_tokens(M, fused, wb) : 0;
    const int64_t tiles = (N + 15) / 16;
    Plan p{};
    for (int per_sm = 2; per_sm >= 1; --per_sm) {
        p.grid = tiles < per_sm * sms ? tiles : per_sm * sms;
        if ((tiles + p.grid - 1) / p.grid > kTileSlots) p.grid = (tiles + kTileSlots - 1) / kTileSlots;
        p.tpc = (tiles + p.grid - 1) / p.grid;
        p.smem = (fixed_smem(static_cast<int>(p.tpc)) + 15) / 16 * 16 + xs_bytes;
        if (per_sm * p.smem <= kSmemCap) break;
    }
    return p;
}

// Weight code widths: WB = 8 (INT8 codes, 16 bytes per lane and block), and
// the W4A8 / W6A8 codes (8 and 12 bytes) that decode onto the INT8 grid: a
// b-bit code c placed in the top bits of a byte is the INT8 value
// c * 2^(8 - b), so the integer sums come out 2^(8 - b) times those of the
// codes and the row scale absorbs the factor (exact: a power of two).
template <int WB>
struct WFmt {
    static_assert(WB == 8 || WB == 6 || WB == 4, "8-, 6- or 4-bit weight codes");
    static constexpr int kWords = WB / 2;       // 32-bit words per lane and block
    static constexpr int kBlockBytes = 64 * WB;  // a block's 16 x 32 codes
    // blocks per load step.  The same for every width: the workloads' K-slices
    // are 6-24 blocks, and steps longer than a slice leave unrolled iterations
    // idle (measured on GB300: 16-block 4-bit steps at K = 4096, 8 of them
    // idle, took the MMA engine from 10.1 to 16.5 us at 12288 x 4096)
    static constexpr int kStep = 8;
    static constexpr float kScale = WB == 8 ? 1.0f : WB == 6 ? 0.25f : 0.0625f;  // 2^-(8 - WB)
};

// The lane's words of one block -> its INT8 A fragment a0..a3 (layouts in include/ck.h).
template <int WB>
__device__ __forceinline__ uint4 decode_fragment(const uint32_t (&v)[WFmt<WB>::kWords]) {
    if constexpr (WB == 8) {
        return make_uint4(v[0], v[1], v[2], v[3]);
    } else if constexpr (WB == 4) {
        // word 0: a0 in the low nibbles, a1 in the high ones; word 1: a2, a3
        constexpr uint32_t hi = 0xF0F0F0F0u;
        return make_uint4((v[0] << 4) & hi, v[0] & hi, (v[1] << 4) & hi, v[1] & hi);
    } else {
        // words 0..2: a0..a2 in bits 2..7 of each byte; a3 in 2-bit pieces in
        // bits 0..1, the low piece in word 0
        constexpr uint32_t top = 0xFCFCFCFCu, low = 0x03030303u;
        return make_uint4(v[0] & top, v[1] & top, v[2] & top,
                          ((v[0] & low) << 2) | ((v[1] & low) << 4) | ((v[2] & low) << 6));
    }
}

__device__ __forceinline__ void mma_s8_16832(int (&d)[4], const uint4 &a, uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// MT (1, 2 or 4): up to MT tokens with four dp4a per token and block (rows g
// and g + 8), summed over the lane's quad at the tile's end; MT = 8 runs the
// INT8 MMA.  FQ = -1: codes xq and scales sx from the quantizer kernel; FQ = 0 / 1:
// the CTA quantizes x (act none / swiglu, group G) itself.  WB: the weight
// code width (WFmt).  S32: y receives the exact int32 sums [M, N] instead of
// the dequantized output (test hook).  early_weights: the weight operands may
// be read before the wait on the kernel ahead.
template <bool XS, int MT, int FQ, int G, int WB = 8, bool S32 = false>
__global__ void __launch_bounds__(kThreads, 2)
gemv_packed_kernel(const int8_t *__restrict__ xq, const float *__restrict__ sx,
                   const __nv_bfloat16 *__restrict__ x, int64_t ldx, int M, int K,
                   const uint8_t *__restrict__ Wp, int N, const __nv_bfloat16 *__restrict__ bias,
                   const __nv_bfloat16 *residual, __nv_bfloat16 *y, int tpc, int early_weights) {
    static_assert(FQ < 0 || XS, "the fused quantizer writes the staged fragments");
    extern __shared__ __align__(16) uint8_t smem[];
    int *red = reinterpret_cast<int *>(smem);             // [tile slot][lane][4]
    int *cnt = red + tpc * 128;                           // [tile slot] warps arrived
    float *ep_sw = reinterpret_cast<float *>(cnt + tpc);  // [tile slot][16] row scales
    float *ep_b = ep_sw + tpc * 16;                       // [tile slot][16] bias
    float *ep_sx = ep_b + tpc * 16;                       // [8] token scales
    float *qred = ep_sx + 8;                              // [warp] fused quantizer maxima
    // activation fragments [block][4 FT]: slot 4 t + c holds codes 32 b + 8 c .. + 7 of token t
    constexpr int FT = MT < 8 ? MT : 8;
    uint2 *xs = reinterpret_cast<uint2 *>(smem + (fixed_smem(tpc) + 15) / 16 * 16);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles = (N + 15) >> 4;
    const int nblk = K >> 5;
    using F = WFmt<WB>;
    constexpr int kSt = F::kStep;
    const size_t tile_bytes = static_cast<size_t>(nblk) * F::kBlockBytes + 64;
    const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * tiles / gridDim.x);
    const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * tiles / gridDim.x);
    const int nslice = min(kWarps, nblk);  // warps with a K-slice
    const int sb = warp < nslice ? warp * nblk / nslice : 0;
    const int se = warp < nslice ? (warp + 1) * nblk / nslice : 0;
    const int spt = (se - sb + kSt - 1) / kSt;  // steps per tile
    const int total = spt * (t1 - t0);          // this warp's steps
    const int grp = lane >> 2, tg4 = lane & 3;

    // step si of tile t0 + k: blocks sb + kSt si ..; this lane's words of
    // each block, loaded into registers
    uint32_t w[kSt][F::kWords];
    auto load_step = [&](int k, int si) {
        const int tt = t0 + k;
        const int b0 = sb + si * kSt;
        const int nb = min(kSt, se - b0);
        const uint8_t *blk = Wp + static_cast<size_t>(tt) * tile_bytes + static_cast<size_t>(b0) * F::kBlockBytes;
#pragma unroll
        for (int j = 0; j < kSt; ++j) {
            const uint8_t *bj = blk + static_cast<size_t>(j) * F::kBlockBytes;
            if constexpr (WB == 8) {
                const uint4 v = j < nb ? __ldg(reinterpret_cast<const uint4 *>(bj) + lane) : make_uint4(0u, 0u, 0u, 0u);
                w[j][0] = v.x; w[j][1] = v.y; w[j][2] = v.z; w[j][3] = v.w;
            } else {
                // words 0 and 1 at 8 lane, word 2 (6-bit) at 256 + 4 lane
                const uint2 v = j < nb ? __ldg(reinterpret_cast<const uint2 *>(bj) + lane) : make_uint2(0u, 0u);
                w[j][0] = v.x; w[j][1] = v.y;
                if constexpr (WB == 6)
                    w[j][2] = j < nb ? __ldg(reinterpret_cast<const uint32_t *>(bj + 256) + lane) : 0u;
            }
        }
    };
    // threads [0, M T) quantize the activation rows in the fused variant (T =
    // round_up(K/32, 32): warp-uniform)
    const int qT = (nblk + 31) & ~31;
    const bool quant_warp = FQ >= 0 && static_cast<int>(threadIdx.x) < M * qT;
    // the weight operands: the first steps' weights and the tiles' dequantization
    // operands.  The warps that will quantize only have L2 fetch their first two
    // steps (a step's blocks are contiguous: one bulk request each) and load them
    // after quantizing, so that no weight registers are live across that code.
    auto start_weights = [&]() {
        if (!quant_warp) {
            if (total > 0) load_step(0, 0);
        } else if (lane == 0) {
            for (int i = 0; i < min(total, 2); ++i) {
                const int tt = t0 + i / spt;
                const int b0 = sb + (i % spt) * kSt;
                const int nb = min(kSt, se - b0);
                prefetch_l2_bulk(Wp + static_cast<size_t>(tt) * tile_bytes + static_cast<size_t>(b0) * F::kBlockBytes,
                                 static_cast<uint32_t>(nb * F::kBlockBytes));
            }
        }
        for (int i = threadIdx.x; i < (t1 - t0) * 16; i += kThreads) {
            const int tt = t0 + i / 16, row = i % 16, n = tt * 16 + row;
            ep_sw[i] = F::kScale * reinterpret_cast<const float *>(Wp + static_cast<size_t>(tt) * tile_bytes +
                                                                   static_cast<size_t>(nblk) * F::kBlockBytes)[row];
            ep_b[i] = (bias != nullptr && n < N) ? __bfloat162float(bias[n]) : 0.0f;
        }
    };
    if (early_weights) start_weights();
    // A kernel queued behind this one may launch now: it waits for our end
    // before it touches anything we read or write.
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < tpc * (128 + 1); i += kThreads) red[i] = 0;
    pdl_wait();  // the activation (codes and scales, or x) comes from the kernel ahead
    if (!early_weights) start_weights();

    if constexpr (FQ < 0) {
        if (threadIdx.x < 8)
            ep_sx[threadIdx.x] = (sx != nullptr && static_cast<int>(threadIdx.x) < M) ? sx[threadIdx.x] : 0.0f;
        if constexpr (XS) {
            // fragment slot (block b, l = 4 t + c): codes 32 b + 8 c .. + 7 of token t
            // (token 0 stands in past M)
            for (int i = threadIdx.x; i < nblk * 4 * FT; i += kThreads) {
                const int b = i / (4 * FT), l = i % (4 * FT), tok = (l >> 2) < M ? (l >> 2) : 0;
                xs[i] = __ldg(reinterpret_cast<const uint2 *>(xq + static_cast<size_t>(tok) * K +
                                                              32 * b + 8 * (l & 3)));
            }
        }
    } else {
        // ---- the CTA quantizes the M activation rows: team r = threads
        // [r T, r T + T) rotates row r, one 32-element unit per thread; the
        // teams exchange their warp maxima through a named barrier of their own
        constexpr int LG = G / 32;
        constexpr int L = LG == 2 ? 1 : LG == 4 ? 2 : 3;
        const int nunits = nblk;
        const int T = qT;
        if (quant_warp) {
            const int qrow = static_cast<int>(threadIdx.x) / T;
            const int qt = static_cast<int>(threadIdx.x) - qrow * T;
            const int q = lane & (LG - 1);
            uint32_t qb[3];
            int cm;
            lane_map<L>(q, qb, cm);
            float2 wq[16];
            {
                // register element e <- position e ^ cm; units past K read unit 0
                const __nv_bfloat16 *src = x + static_cast<int64_t>(qrow) * ldx +
                                           static_cast<int64_t>(qt < nunits ? qt : 0) * 32;
                uint32_t ra[16], rb[16];
                if constexpr (L < 3) {
#pragma unroll
                    for (int rc = 0; rc < 4; ++rc) {
                        const int pc = rc ^ (cm >> 3);
                        const uint4 va = __ldg(reinterpret_cast<const uint4 *>(src + 8 * pc));
                        ra[4 * rc] = va.x; ra[4 * rc + 1] = va.y; ra[4 * rc + 2] = va.z; ra[4 * rc + 3] = va.w;
                        if constexpr (FQ == static_cast<int>(Act::kSwiglu)) {
                            const uint4 vb = __ldg(reinterpret_cast<const uint4 *>(src + K + 8 * pc));
                            rb[4 * rc] = vb.x; rb[4 * rc + 1] = vb.y; rb[4 * rc + 2] = vb.z; rb[4 * rc + 3] = vb.w;
                        }
                    }
                } else {
#pragma unroll
                    for (int rh = 0; rh < 8; ++rh) {
                        const int ph = rh ^ (cm >> 2);
                        const uint2 va = __ldg(reinterpret_cast<const uint2 *>(src + 4 * ph));
                        ra[2 * rh] = va.x; ra[2 * rh + 1] = va.y;
                        if constexpr (FQ == static_cast<int>(Act::kSwiglu)) {
                            const uint2 vb = __ldg(reinterpret_cast<const uint2 *>(src + K + 4 * ph));
                            rb[2 * rh] = vb.x; rb[2 * rh + 1] = vb.y;
                        }
                    }
                }
                rotate_unit<FQ, L>(ra, rb, qb, wq);
            }
            float amax = qt < nunits ? unit_absmax(wq) : 0.0f;
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
            if (lane == 0) qred[warp] = amax;
            named_bar_sync(1, M * T);
            amax = 0.0f;
            for (int ww = 0; ww < (T >> 5); ++ww) amax = fmaxf(amax, qred[qrow * (T >> 5) + ww]);
            constexpr float c = static_cast<float>(InvSqrtG<G>::v);
            const float s = __fdiv_rn(amax * c, 127.0f);  // max |f32(v / sqrt g)| / 127
            if (qt == 0) ep_sx[qrow] = s;
            if (qt < nunits)
                quantize_unit<G, FT == 1 ? kOutFrag1 : FT == 2 ? kOutFrag2 : FT == 4 ? kOutFrag4 : kOutFrag8>(
                    wq, s, __frcp_rn(s), scale_in_range(amax), qb, nullptr,
                    reinterpret_cast<int8_t *>(xs) + 32 * qrow, static_cast<int64_t>(qt - q) * 32 + cm);
            // from L2 by now; defined on every path, so that no earlier weight
            // registers stay live across the code above
            if (total > 0) {
                load_step(0, 0);
            } else {
#pragma unroll
                for (int j = 0; j < kSt; ++j)
#pragma unroll
                    for (int q = 0; q < F::kWords; ++q) w[j][q] = 0u;
            }
        }
        if constexpr (MT == 8) {
            // the MMA reads all eight token slots: zero those of tokens past M
            for (int i = threadIdx.x; i < nblk * 32; i += kThreads)
                if (((i >> 2) & 7) >= M) xs[i] = make_uint2(0u, 0u);
        }
        if (threadIdx.x < 8 && static_cast<int>(threadIdx.x) >= M) ep_sx[threadIdx.x] = 0.0f;
    }
    __syncthreads();

    // this lane's activation codes when they are read through L1 (K past the staging limit)
    const int8_t *xrow = XS ? nullptr : xq + static_cast<size_t>(grp < M ? grp : 0) * K + 8 * tg4;
    int acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
    constexpr int kCh = MT >= 4 ? 1 : 2;  // independent dp4a chains per token and row
    int dacc[kCh][MT < 8 ? MT : 1][2] = {};  // [chain][token][row g, row g + 8]
    // step i = the warp's tile k, step si of it (counted, not divided out)
    int k = 0, si = 0;
    for (int i = 0; i < total; ++i) {
        const int tt = t0 + k;
        const int b0 = sb + si * kSt;
        const int nb = min(kSt, se - b0);
#pragma unroll
        for (int j = 0; j < kSt; ++j) {
            if (j < nb) {
                const uint4 wf = decode_fragment<WB>(w[j]);
                if constexpr (MT < 8) {
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        // token t's codes 32 b + 8 c .. + 7 (token 0 stands in past M)
                        const uint2 xf = XS ? xs[(b0 + j) * 4 * FT + 4 * t + tg4]
                                            : __ldg(reinterpret_cast<const uint2 *>(
                                                  xq + static_cast<size_t>(t < M ? t : 0) * K +
                                                  32 * (b0 + j) + 8 * tg4));
                        int &a = dacc[j % kCh][t][0], &c = dacc[j % kCh][t][1];
                        a = __dp4a(static_cast<int>(wf.x), static_cast<int>(xf.x), a);
                        a = __dp4a(static_cast<int>(wf.z), static_cast<int>(xf.y), a);
                        c = __dp4a(static_cast<int>(wf.y), static_cast<int>(xf.x), c);
                        c = __dp4a(static_cast<int>(wf.w), static_cast<int>(xf.y), c);
                    }
                } else {
                    const uint2 xf = XS ? xs[(b0 + j) * 32 + lane]
                                        : __ldg(reinterpret_cast<const uint2 *>(xrow + 32 * (b0 + j)));
                    mma_s8_16832(acc[j & 1], wf, xf.x, xf.y);
                }
            }
        }
        const bool tile_done = si == spt - 1;
        si = tile_done ? 0 : si + 1;
        k += tile_done ? 1 : 0;
        if (i + 1 < total) load_step(k, si);
        if (tile_done) {
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
                    if constexpr (S32) {
                        // the exact sums themselves (test hook): on the INT8 grid, so
                        // 2^(8-b) times the b-bit codes' sums; y is int32 [M, N]
                        if (tok < M && n < N) reinterpret_cast<int32_t *>(y)[static_cast<size_t>(tok) * N + n] = tot;
                    } else if (tok < M && n < N) {
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

}  // namespace gv
}  // namespace ck
