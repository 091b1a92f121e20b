// gemm_epilogue.cuh -- the dequant epilogue of the tcgen05 GEMMs (one-SM and
// CTA-pair kernels):
//
//   y[m, n] = bf16( (f32(acc[m, n]) * sx[m] * sw[n] + bias[n]) + residual[m, n] )
// (comfy-kitchen PR #277, "Summary": per-token and per-output-row scales applied
// to the exact int32 sums, then the bias).
//
// Eight epilogue warps (256 threads, named barrier 1) share one output tile of
// 128 rows x TN columns; thread (warp w, lane l) holds the int32 sums of row
// 32 * (w % 4) + l over one half (TN / 2 columns) of the tile.
//
//  - The tile's column scales and bias are read from global memory once, at
//    the start of the tile, into shared memory (TN floats each), while the
//    tensor core is still producing the tile; the dequant reads them as
//    shared-memory broadcasts instead of one dependent global load per eight
//    columns at the end of the tile; each thread's token scale is read at the
//    start of the tile as well (the kernels pass it in).
//  - Stores are coalesced by a 4 x 4 transpose of 16-byte pieces within each
//    quad of lanes (two shuffle rounds): after it, one store instruction of
//    the warp writes 64 contiguous bytes in each of 8 rows instead of
//    16 bytes in each of 32 rows (every width; the GLU output keeps row-owner
//    stores for 128-column halves, where the exchange spills ~490 bytes).
//  - The residual is read by the row's owner, each 16-byte piece of a
//    32-column group before any store of the group, so it may be the output
//    itself.
//
// The SwiGLU output (kOutGlu; sglang PR #44196, "Motivation": silu(gate) * up
// formed in FP32 from the bf16 gate|up linear): the weight rows come
// interleaved -- column 2j of the tile is gate row j, column 2j + 1 up row j
// of the [gate | up] weight, whose scales and bias are staged from their
// original places -- and each thread turns the bf16 pair it dequantizes into
//   a[m, j] = silu(f32(gate)) * f32(up)    (f32, stored [M, N / 2])
// with the activation quantizer's own silu_mul, so that the down linear's
// quantizer sees bit for bit the product it would have formed itself.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_core.cuh"

namespace ck {
namespace ep {

constexpr int kThreads = 256;  // epilogue warps 2..9
constexpr int kBarId = 1;

// Shared-memory bytes for the staged scales and bias of a tile of tn columns.
__host__ __device__ constexpr int staging_bytes(int tn) { return tn * 8; }

// All epilogue threads have finished reading the previous tile's staging.
__device__ __forceinline__ void sync() { named_bar_sync(kBarId, kThreads); }

// Barrier that also makes `ok` uniform: true only if it is true in every
// epilogue thread.  It publishes the staged scales as well.
__device__ __forceinline__ bool sync_all_ok(bool ok) {
    return !named_bar_or(kBarId, kThreads, !ok);
}

// Columns n_base .. n_base + tn - 1 of sw and bias into shared memory (zero
// past N); thread t (0..255) of the epilogue fills column t.
__device__ __forceinline__ void stage(float *ssw, float *sb, int t, int tn, int n_base, int N,
                                      const float *__restrict__ sw,
                                      const __nv_bfloat16 *__restrict__ bias) {
    if (t < tn) {
        const int n = n_base + t;
        const bool in = n < N;
        ssw[t] = in ? __ldg(sw + n) : 0.f;
        sb[t] = (in && bias != nullptr) ? __bfloat162float(bias[n]) : 0.f;
    }
}

// stage() for interleaved gate / up columns (kOutGlu): tile column t is
// [gate | up] row (n_base + t) / 2 + (t odd ? N / 2 : 0); N is the
// interleaved width (2 I), n_base even.
__device__ __forceinline__ void stage_glu(float *ssw, float *sb, int t, int tn, int n_base, int N,
                                          const float *__restrict__ sw,
                                          const __nv_bfloat16 *__restrict__ bias) {
    if (t < tn) {
        const int n = n_base + t;
        const bool in = n < N;
        const int src = (n >> 1) + ((n & 1) ? (N >> 1) : 0);
        ssw[t] = in ? __ldg(sw + src) : 0.f;
        sb[t] = (in && bias != nullptr) ? __bfloat162float(bias[src]) : 0.f;
    }
}

// Eight columns of one row: acc * s_x * sw + b + r, packed to bf16 pairs
// (r: eight bf16 residual values, zero when there is none).
__device__ __forceinline__ void dequant8(const int32_t *acc, float s_x, const float *w,
                                         const float *b, const uint4 ru, uint32_t *pk) {
    const float4 w0 = *reinterpret_cast<const float4 *>(w);
    const float4 w1 = *reinterpret_cast<const float4 *>(w + 4);
    const float4 b0 = *reinterpret_cast<const float4 *>(b);
    const float4 b1 = *reinterpret_cast<const float4 *>(b + 4);
    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const uint32_t rw[4] = {ru.x, ru.y, ru.z, ru.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float r0 = __uint_as_float(rw[e] << 16), r1 = __uint_as_float(rw[e] & 0xffff0000u);
        const float y0 = (static_cast<float>(acc[2 * e]) * s_x * wv[2 * e] + bv[2 * e]) + r0;
        const float y1 = (static_cast<float>(acc[2 * e + 1]) * s_x * wv[2 * e + 1] + bv[2 * e + 1]) + r1;
        const __nv_bfloat162 v = __floats2bfloat162_rn(y0, y1);
        pk[e] = *reinterpret_cast<const uint32_t *>(&v);
    }
}

// P holds four 16-byte pieces (words 4k .. 4k+3 = piece k) of the row owned by
// quad lane qi.  Afterwards words 4k .. 4k+3 hold piece qi of the row owned by
// quad lane k.  Round one swaps the off-diagonal 2 x 2 blocks with lane qi ^ 2,
// round two the off-diagonal pieces of each block with lane qi ^ 1.
__device__ __forceinline__ void quad_transpose(uint32_t (&P)[16], int qi) {
    const bool b1 = (qi & 2) != 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t got = __shfl_xor_sync(0xffffffffu, b1 ? P[w] : P[w + 8], 2);
        if (b1)
            P[w] = got;
        else
            P[w + 8] = got;
    }
    const bool b0 = (qi & 1) != 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int lo = 8 * e + w, hi = 8 * e + 4 + w;
            const uint32_t got = __shfl_xor_sync(0xffffffffu, b0 ? P[lo] : P[hi], 1);
            if (b0)
                P[lo] = got;
            else
                P[hi] = got;
        }
    }
}

// Dequantize and store this thread's half-row of the tile.
//   row0   first row of the warp (the thread's row is row0 + lane)
//   s_x    the row's token scale (read at the start of the tile: a global load
//          at the end would add its latency to the tile's tail)
//   n0     first column of the half; ssw/sb point at the staged values of n0
// Requires N % 8 == 0 (each 8-column piece is wholly inside or outside).
// Half-rows of 128 columns take the exchange too, although with 128 int32
// sums live ptxas then spills ~190 bytes a thread: measured on GB300 the
// coalesced stores still win (256-wide tiles 3-6 % faster at 2048 x 3072 ->
// 2048 and 4096^3, 17 % at 2048 x 1024 -> 3072).
template <int kCols>
__device__ __forceinline__ void dequant_store(const int32_t (&acc)[kCols], int row0, int lane, int M,
                                              int n0, int N, float s_x, const float *ssw,
                                              const float *sb, const __nv_bfloat16 *residual,
                                              __nv_bfloat16 *out) {
    static_assert(kCols % 16 == 0, "half-tile width must be a multiple of 16");
    constexpr bool kExchange = kCols <= 128;
    constexpr int kGroups = kExchange ? kCols / 32 : 0;  // 32-column groups
    const int m = row0 + lane;
    const bool row_in = m < M;
    const __nv_bfloat16 *res_row =
        residual != nullptr ? residual + static_cast<int64_t>(m) * N + n0 : nullptr;
    // the residual piece at column c of the half (read before any store of its group)
    auto res = [&](int c) {
        return (res_row != nullptr && row_in && n0 + c < N)
                   ? *reinterpret_cast<const uint4 *>(res_row + c)
                   : make_uint4(0u, 0u, 0u, 0u);
    };
    const int qi = lane & 3;
    const int quad_row0 = row0 + (lane & ~3);
#pragma unroll
    for (int grp = 0; grp < kGroups; ++grp) {
        uint32_t P[16];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int c = 32 * grp + 8 * p;
            dequant8(&acc[c], s_x, ssw + c, sb + c, res(c), &P[4 * p]);
        }
        quad_transpose(P, qi);
        const int n = n0 + 32 * grp + 8 * qi;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int mr = quad_row0 + k;
            if (mr < M && n < N)
                *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(mr) * N + n) =
                    make_uint4(P[4 * k], P[4 * k + 1], P[4 * k + 2], P[4 * k + 3]);
        }
    }
    // what is left (a 128-column half-row, else the last 16 columns of a
    // 112-column one): the row's owner stores it, 8 columns at a time
#pragma unroll
    for (int c = 32 * kGroups; c < kCols; c += 8) {
        if (row_in && n0 + c < N) {
            uint32_t pk[4];
            dequant8(&acc[c], s_x, ssw + c, sb + c, res(c), pk);
            *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(m) * N + n0 + c) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
    }
}

// kOutGlu: this thread's half-row of interleaved gate / up sums ->
// a = silu(gate) * up, f32, kCols / 2 values at out[m, n0 / 2 ..] (out is
// [M, N / 2]).  gate and up are the bf16 values dequant8 gives the plain
// output (no residual), so a is the product the swiglu quantizer forms from
// that output.  Stores as dequant_store's: per 32-column group (16 products,
// 64 bytes of the row) the quad transpose leaves each lane one 16-byte piece
// of four rows, so a warp's store covers 64 contiguous bytes of 8 rows.
template <int kCols>
__device__ __forceinline__ void glu_store(const int32_t (&acc)[kCols], int row0, int lane, int M,
                                          int n0, int N, float s_x, const float *ssw,
                                          const float *sb, float *out) {
    static_assert(kCols % 16 == 0, "half-tile width must be a multiple of 16");
    constexpr bool kExchange = kCols < 128;
    constexpr int kGroups = kExchange ? kCols / 32 : 0;
    const int m = row0 + lane;
    const int64_t ldo = N >> 1;
    // the four products of the 8-column piece at column c of the half
    auto products = [&](int c, uint32_t *dst) {
        uint32_t pk[4];
        dequant8(&acc[c], s_x, ssw + c, sb + c, make_uint4(0u, 0u, 0u, 0u), pk);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            dst[e] = __float_as_uint(
                qc::silu_mul(__uint_as_float(pk[e] << 16), __uint_as_float(pk[e] & 0xffff0000u)));
    };
    const int qi = lane & 3;
    const int quad_row0 = row0 + (lane & ~3);
#pragma unroll
    for (int grp = 0; grp < kGroups; ++grp) {
        uint32_t P[16];
#pragma unroll
        for (int p = 0; p < 4; ++p) products(32 * grp + 8 * p, &P[4 * p]);
        quad_transpose(P, qi);
        const int n = n0 + 32 * grp + 8 * qi;  // the piece's first interleaved column
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int mr = quad_row0 + k;
            if (mr < M && n < N)
                *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(mr) * ldo + (n >> 1)) =
                    make_uint4(P[4 * k], P[4 * k + 1], P[4 * k + 2], P[4 * k + 3]);
        }
    }
    // the rest: the row's owner stores it, four products at a time
#pragma unroll
    for (int c = 32 * kGroups; c < kCols; c += 8) {
        if (m < M && n0 + c < N) {
            uint32_t a[4];
            products(c, a);
            *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(m) * ldo + ((n0 + c) >> 1)) =
                make_uint4(a[0], a[1], a[2], a[3]);
        }
    }
}

}  // namespace ep
}  // namespace ck
