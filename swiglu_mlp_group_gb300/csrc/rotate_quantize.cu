// rotate_quantize.cu -- fused group-Hadamard rotation + per-row absmax INT8
// quantization (with the optional SwiGLU input activation).
//
// Computes, for every row of x (activations, or weight rows offline):
//   v     = x                       (act none)  or  silu(gate) * up in f32 (act swiglu)
//   v_rot = v H, H = blockdiag(H_g), H_g the Sylvester Hadamard / sqrt(g)
//   s     = max_k |v_rot[k]| / 127,  q[k] = clamp(rne(v_rot[k] / s), -127, 127)
// as in comfy-kitchen PR #277 "The key observation" (x_rot = x @ H, the GEMM
// stays in the rotated basis), the per-row INT8 grid of its "Notes for the
// reviewer", the weight quantizer of the sglang PR #35994 report
// (kitchen_int8.py: per_channel, convrot_groupsize, stochastic_rounding=0),
// and the SwiGLU quantizer of sglang PR #44196 "Motivation".
//
// Mapping: a row is handled by a team of T threads (a multiple of 32).  The
// row is split into 8-element chunks (16 bytes of bf16); thread t owns chunks
// t, t + T, ..., so every load instruction of a warp reads consecutive
// 16-byte pieces.  A group of g elements is g/8 consecutive chunks, i.e.
// g/8 consecutive lanes of one warp: the Walsh-Hadamard butterflies run in
// registers for strides 1, 2, 4 and through __shfl_xor_sync for strides
// 8 .. g/2.  The row absmax is a warp shuffle reduction plus one shared-memory
// exchange between the team's warps.  HBM-bound: one read of x, one write of
// the codes.
//
// Precision: activations are rotated in f32 (on the hot path).  Weights are
// quantized once, offline, so their rotation runs in float64 and is rounded
// once to f32 -- the definition the reference arithmetic uses -- which makes
// the weight codes independent of the butterfly order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ck {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xffff0000u);
    v[4] = __uint_as_float(u.z << 16);
    v[5] = __uint_as_float(u.z & 0xffff0000u);
    v[6] = __uint_as_float(u.w << 16);
    v[7] = __uint_as_float(u.w & 0xffff0000u);
}

__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// silu(z) * u in f32, silu(z) = z / (1 + exp(-z)).
__device__ __forceinline__ float silu_mul(float z, float u) {
    return __fdiv_rn(z, 1.0f + expf(-z)) * u;
}

// 1/sqrt(g), as a double (rounded to f32 where the rotation runs in f32)
template <int G>
struct InvSqrtG;
template <> struct InvSqrtG<64> { static constexpr double v = 0.125; };
template <> struct InvSqrtG<128> { static constexpr double v = 0.08838834764831845; };
template <> struct InvSqrtG<256> { static constexpr double v = 0.0625; };

template <typename TIn, typename TAcc, int ACT, int G, int R, int OUT>
__global__ void __launch_bounds__(512)
rotate_quantize_kernel(const TIn *__restrict__ x, int M, int K, int64_t ldx,
                       int8_t *__restrict__ q8, __half *__restrict__ q16,
                       float *__restrict__ scale, int T) {
    extern __shared__ float red[];  // [blockDim.y][T / 32] warp maxima
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.y + threadIdx.y;
    const bool row_ok = row < M;
    const int nchunks = K >> 3;

    TAcc v[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int c = t + r * T;
        float in[8];
        if (row_ok && c < nchunks) {
            const TIn *src = x + row * ldx + static_cast<int64_t>(c) * 8;
            if constexpr (ACT == static_cast<int>(Act::kSwiglu)) {
                float up[8];
                load8(src, in);
                load8(src + K, up);
#pragma unroll
                for (int e = 0; e < 8; ++e) in[e] = silu_mul(in[e], up[e]);
            } else {
                load8(src, in);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) in[e] = 0.0f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) v[r][e] = static_cast<TAcc>(in[e]);
    }
    // Our reads are issued: a dependent kernel may start its prologue.
    pdl_launch_dependents();

    // Walsh-Hadamard butterflies (u, w) -> (u + w, u - w), natural order.
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if ((e & h) == 0) {
                    const TAcc a = v[r][e], b = v[r][e + h];
                    v[r][e] = a + b;
                    v[r][e + h] = a - b;
                }
            }
        }
    }
#pragma unroll
    for (int m = 1; m < G / 8; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const TAcc p = __shfl_xor_sync(kFull, v[r][e], m);
                v[r][e] = upper ? (p - v[r][e]) : (v[r][e] + p);
            }
        }
    }

    // normalise and round to f32 (once, for the float64 path)
    float vr[R][8];
    float amax = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            vr[r][e] = static_cast<float>(v[r][e] * static_cast<TAcc>(InvSqrtG<G>::v));
            amax = fmaxf(amax, fabsf(vr[r][e]));
        }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
    const int nw = T >> 5;
    if (lane == 0) red[threadIdx.y * nw + (t >> 5)] = amax;
    __syncthreads();
    amax = 0.0f;
    for (int w = 0; w < nw; ++w) amax = fmaxf(amax, red[threadIdx.y * nw + w]);
    const float s = __fdiv_rn(amax, 127.0f);
    if (t == 0 && row_ok) scale[row] = s;
    if (!row_ok) return;

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int c = t + r * T;
        if (c >= nchunks) continue;
        int qi[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float qq = (s == 0.0f) ? 0.0f : rintf(__fdiv_rn(vr[r][e], s));
            qq = fminf(fmaxf(qq, -127.0f), 127.0f);
            qi[e] = static_cast<int>(qq);
        }
        const int64_t off = row * K + static_cast<int64_t>(c) * 8;
        if constexpr ((OUT & kOutI8) != 0) {
            uint2 pk;
            pk.x = (qi[0] & 0xff) | ((qi[1] & 0xff) << 8) | ((qi[2] & 0xff) << 16) |
                   (static_cast<unsigned>(qi[3] & 0xff) << 24);
            pk.y = (qi[4] & 0xff) | ((qi[5] & 0xff) << 8) | ((qi[6] & 0xff) << 16) |
                   (static_cast<unsigned>(qi[7] & 0xff) << 24);
            *reinterpret_cast<uint2 *>(q8 + off) = pk;
        }
        if constexpr ((OUT & kOutF16) != 0) {
            uint4 pk;
            pk.x = __half_as_ushort(__int2half_rn(qi[0])) |
                   (static_cast<unsigned>(__half_as_ushort(__int2half_rn(qi[1]))) << 16);
            pk.y = __half_as_ushort(__int2half_rn(qi[2])) |
                   (static_cast<unsigned>(__half_as_ushort(__int2half_rn(qi[3]))) << 16);
            pk.z = __half_as_ushort(__int2half_rn(qi[4])) |
                   (static_cast<unsigned>(__half_as_ushort(__int2half_rn(qi[5]))) << 16);
            pk.w = __half_as_ushort(__int2half_rn(qi[6])) |
                   (static_cast<unsigned>(__half_as_ushort(__int2half_rn(qi[7]))) << 16);
            *reinterpret_cast<uint4 *>(q16 + off) = pk;
        }
    }
}

template <typename TIn, typename TAcc, int ACT, int G, int R, int OUT>
cudaError_t launch_t(const void *x, int64_t M, int64_t K, int64_t ldx, int8_t *q8, void *q16,
                     float *scale, int T, int rows_per_cta, const LaunchCtx &ctx) {
    const dim3 block(T, rows_per_cta);
    const dim3 grid(static_cast<unsigned>((M + rows_per_cta - 1) / rows_per_cta));
    const size_t smem = sizeof(float) * static_cast<size_t>(rows_per_cta) * (T / 32);
    rotate_quantize_kernel<TIn, TAcc, ACT, G, R, OUT><<<grid, block, smem, ctx.stream>>>(
        static_cast<const TIn *>(x), static_cast<int>(M), static_cast<int>(K), ldx, q8,
        static_cast<__half *>(q16), scale, T);
    return cudaGetLastError();
}

template <typename TIn, typename TAcc, int ACT, int G, int OUT>
cudaError_t dispatch_r(int R, const void *x, int64_t M, int64_t K, int64_t ldx, int8_t *q8,
                       void *q16, float *scale, int T, int rpc, const LaunchCtx &ctx) {
    switch (R) {
        case 1: return launch_t<TIn, TAcc, ACT, G, 1, OUT>(x, M, K, ldx, q8, q16, scale, T, rpc, ctx);
        case 2: return launch_t<TIn, TAcc, ACT, G, 2, OUT>(x, M, K, ldx, q8, q16, scale, T, rpc, ctx);
        case 4: return launch_t<TIn, TAcc, ACT, G, 4, OUT>(x, M, K, ldx, q8, q16, scale, T, rpc, ctx);
        default: return launch_t<TIn, TAcc, ACT, G, 8, OUT>(x, M, K, ldx, q8, q16, scale, T, rpc, ctx);
    }
}

template <typename TIn, typename TAcc, int ACT, int OUT>
cudaError_t dispatch_g(int g, int R, const void *x, int64_t M, int64_t K, int64_t ldx,
                       int8_t *q8, void *q16, float *scale, int T, int rpc,
                       const LaunchCtx &ctx) {
    switch (g) {
        case 64: return dispatch_r<TIn, TAcc, ACT, 64, OUT>(R, x, M, K, ldx, q8, q16, scale, T, rpc, ctx);
        case 128: return dispatch_r<TIn, TAcc, ACT, 128, OUT>(R, x, M, K, ldx, q8, q16, scale, T, rpc, ctx);
        case 256: return dispatch_r<TIn, TAcc, ACT, 256, OUT>(R, x, M, K, ldx, q8, q16, scale, T, rpc, ctx);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_rotate_quantize(const void *x, bool x_f32, Act act, int g, int64_t M,
                                   int64_t K, int64_t ldx, int8_t *q8, void *q16, float *scale,
                                   const LaunchCtx &ctx, bool f64_rotation) {
    if (M <= 0) return cudaSuccess;
    const int64_t nchunks = K / 8;
    int R = 1;
    while ((nchunks + R - 1) / R > 128 && R < 8) R *= 2;
    const int T = static_cast<int>(((nchunks + R - 1) / R + 31) / 32 * 32);
    if (T > 512) return cudaErrorInvalidValue;
    const int rpc = T >= 256 ? 1 : 256 / T;
    const int out = (q8 ? kOutI8 : 0) | (q16 ? kOutF16 : 0);
    if (f64_rotation) {
        // offline weight quantization: int8 codes only, float64 rotation
        if (act != Act::kNone || out != kOutI8) return cudaErrorInvalidValue;
        if (x_f32)
            return dispatch_g<float, double, 0, kOutI8>(g, R, x, M, K, ldx, q8, q16, scale, T, rpc, ctx);
        return dispatch_g<__nv_bfloat16, double, 0, kOutI8>(g, R, x, M, K, ldx, q8, q16, scale, T,
                                                            rpc, ctx);
    }
    if (x_f32) return cudaErrorInvalidValue;
    if (act == Act::kNone) {
        if (out == kOutI8)
            return dispatch_g<__nv_bfloat16, float, 0, kOutI8>(g, R, x, M, K, ldx, q8, q16, scale, T,
                                                               rpc, ctx);
        if (out == kOutF16)
            return dispatch_g<__nv_bfloat16, float, 0, kOutF16>(g, R, x, M, K, ldx, q8, q16, scale,
                                                                T, rpc, ctx);
        return cudaErrorInvalidValue;
    }
    if (out == kOutI8)
        return dispatch_g<__nv_bfloat16, float, 1, kOutI8>(g, R, x, M, K, ldx, q8, q16, scale, T,
                                                           rpc, ctx);
    if (out == kOutF16)
        return dispatch_g<__nv_bfloat16, float, 1, kOutF16>(g, R, x, M, K, ldx, q8, q16, scale, T,
                                                            rpc, ctx);
    return cudaErrorInvalidValue;
}

}  // namespace ck
