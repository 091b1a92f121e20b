// rotate_quantize.cu -- fused group-Hadamard rotation + per-row absmax INT8
// quantization (with the optional SwiGLU input activation).
//
// Computes, for every row of x (activations, or weight rows offline):
//   v     = x                       (act none)  or  silu(gate) * up in f32 (act swiglu,
//           or that product read back in f32 after the gate|up GEMM formed it)
//   v_rot = v H, H = blockdiag(H_g), H_g the Sylvester Hadamard / sqrt(g)
//   s     = max_k |v_rot[k]| / 127,  q[k] = clamp(rne(v_rot[k] / s), -127, 127)
// as in comfy-kitchen PR #277 "The key observation" (x_rot = x @ H, the GEMM
// stays in the rotated basis), the per-row INT8 grid of its "Notes for the
// reviewer", the weight quantizer of the sglang PR #35994 report
// (kitchen_int8.py: per_channel, convrot_groupsize, stochastic_rounding=0),
// and the SwiGLU quantizer of sglang PR #44196 "Motivation".
//
// Mapping: a row is handled by a team of T threads (a multiple of 32).  The
// row is cut into units of 32 contiguous elements; thread t owns units t,
// t + T, ... (U of them).  A group of g elements is g/32 consecutive units,
// i.e. g/32 consecutive lanes of one warp: the Walsh-Hadamard butterflies run
// in registers for strides 1..16 and as half-exchange shuffle stages for
// strides 32..g/2.  The row absmax is a warp shuffle reduction plus one
// shared-memory exchange between the team's warps.  HBM-bound: one read of x,
// one write of the codes.
//
// Activations rotate in f32 with the 1/sqrt(g) normalisation folded into the
// quantization: the codes are rint(v_rot * f), f = f32(1/sqrt g) * f32(1/s),
// within a few ulps of z / s (the device pieces of that path, and their
// description, are in quant_core.cuh).
//
// Weights (offline) are rotated in float64 and rounded once to f32 -- the
// definition the reference arithmetic uses -- which makes the weight codes
// independent of the butterfly order; they are then divided by the scale.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "quant_core.cuh"

namespace ck {
namespace {

using namespace qc;


// Raw bytes of one 8-element chunk (two 16-byte words: f32 input, or the
// gate and up halves of a swiglu input; one word for plain bf16).
struct RawChunk {
    uint4 a, b;
};

template <typename TIn, int ACT>
__device__ __forceinline__ void load_raw(const TIn *src, int64_t up_off, RawChunk &r) {
    r.a = __ldg(reinterpret_cast<const uint4 *>(src));
    if constexpr (sizeof(TIn) == 4) r.b = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
    if constexpr (ACT == 1) r.b = __ldg(reinterpret_cast<const uint4 *>(src + up_off));
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&v)[8]) {
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xffff0000u);
    v[4] = __uint_as_float(u.z << 16);
    v[5] = __uint_as_float(u.z & 0xffff0000u);
    v[6] = __uint_as_float(u.w << 16);
    v[7] = __uint_as_float(u.w & 0xffff0000u);
}


template <typename TIn, typename TAcc, int ACT, int G, int U, int OUT>
__global__ void __launch_bounds__(512)
rotate_quantize_kernel(const TIn *__restrict__ x, int M, int K, int64_t ldx,
                       int8_t *__restrict__ q8, __half *__restrict__ q16,
                       float *__restrict__ scale, int T, int qmax) {
    extern __shared__ float red[];  // [2][blockDim.y][T / 32] warp maxima (double-buffered)
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int nunits = K >> 5;
    const int nw = T >> 5;
    const int64_t row_step = static_cast<int64_t>(gridDim.x) * blockDim.y;

    // The CTA walks rows base, base + row_step, ...; the raw input of the next
    // row is loaded while the current one is transformed.
    RawChunk raw[U][4];
    auto issue_loads = [&](int64_t r) {
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int u = t + j * T;
            if (r < M && u < nunits) {
                const TIn *src = x + r * ldx + static_cast<int64_t>(u) * 32;
#pragma unroll
                for (int c = 0; c < 4; ++c) load_raw<TIn, ACT>(src + 8 * c, K, raw[j][c]);
            }
        }
    };
    int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.y + threadIdx.y;
    issue_loads(row);
    // Our first reads are issued: a dependent kernel may start its prologue.
    pdl_launch_dependents();

    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.y, it = 0; base < M;
         base += row_step, row += row_step, ++it) {
    const bool row_ok = row < M;
    float *redb = red + (it & 1) * blockDim.y * nw;

    TAcc v[U][32];
#pragma unroll
    for (int j = 0; j < U; ++j) {
        const bool ok = row_ok && t + j * T < nunits;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float in[8];
            if (ok) {
                if constexpr (sizeof(TIn) == 4) {
                    const uint4 a = raw[j][c].a, b = raw[j][c].b;
                    in[0] = __uint_as_float(a.x); in[1] = __uint_as_float(a.y);
                    in[2] = __uint_as_float(a.z); in[3] = __uint_as_float(a.w);
                    in[4] = __uint_as_float(b.x); in[5] = __uint_as_float(b.y);
                    in[6] = __uint_as_float(b.z); in[7] = __uint_as_float(b.w);
                } else if constexpr (ACT == static_cast<int>(Act::kSwiglu)) {
                    float up[8];
                    bf16x8_to_f32(raw[j][c].a, in);
                    bf16x8_to_f32(raw[j][c].b, up);
#pragma unroll
                    for (int e = 0; e < 8; ++e) in[e] = silu_mul(in[e], up[e]);
                } else {
                    bf16x8_to_f32(raw[j][c].a, in);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) in[e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) v[j][8 * c + e] = static_cast<TAcc>(in[e]);
        }
    }
    issue_loads(row + row_step);

    // Walsh-Hadamard butterflies (a, b) -> (a + b, a - b), natural order.
#pragma unroll
    for (int j = 0; j < U; ++j) {
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                if ((e & h) == 0) {
                    const TAcc a = v[j][e], b = v[j][e + h];
                    v[j][e] = a + b;
                    v[j][e + h] = a - b;
                }
            }
        }
    }
#pragma unroll
    for (int m = 1; m < G / 32; m <<= 1) {
        // lower lane: mine + partner's; upper lane: partner's - mine
        const TAcc sgn = (lane & m) ? TAcc(-1) : TAcc(1);
#pragma unroll
        for (int j = 0; j < U; ++j) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const TAcc p = __shfl_xor_sync(kFull, v[j][e], m);
                v[j][e] = fma(sgn, v[j][e], p);
            }
        }
    }

    static_assert(sizeof(TAcc) == 8, "the offline weight path rotates in float64");
    {
        // ---- weights: normalise in float64, round once to f32, divide
        float vr[U][32];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < U; ++j) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                vr[j][e] = static_cast<float>(v[j][e] * InvSqrtG<G>::v);
                amax = fmaxf(amax, fabsf(vr[j][e]));
            }
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
        if (lane == 0) redb[threadIdx.y * nw + (t >> 5)] = amax;
        __syncthreads();
        amax = 0.0f;
        for (int w = 0; w < nw; ++w) amax = fmaxf(amax, redb[threadIdx.y * nw + w]);
        // codes of at most qmax in magnitude: 127 (INT8), 31 (6-bit), 7 (4-bit)
        const float qm = static_cast<float>(qmax);
        const float s = __fdiv_rn(amax, qm);
        if (t == 0 && row_ok) scale[row] = s;
        if (!row_ok) continue;
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int u = t + j * T;
            if (u >= nunits) continue;
            uint32_t pk[8];
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
                uint32_t word = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    float qq = (s == 0.0f) ? 0.0f : rintf(__fdiv_rn(vr[j][4 * e4 + b], s));
                    qq = fminf(fmaxf(qq, -qm), qm);
                    word |= (static_cast<uint32_t>(static_cast<int>(qq)) & 0xffu) << (8 * b);
                }
                pk[e4] = word;
            }
            uint4 *dst = reinterpret_cast<uint4 *>(q8 + row * K + static_cast<int64_t>(u) * 32);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
    }
    }  // row loop
}


// ---- one row per team, U units per lane (U = 2 beyond K = 16384)
template <int ACT, int G, int U, int OUT>
__global__ void __launch_bounds__(512, U == 1 ? 2 : 1)
rotate_quantize_act_kernel(const __nv_bfloat16 *__restrict__ x, int M, int K, int64_t ldx,
                           int8_t *__restrict__ q8, __half *__restrict__ q16,
                           float *__restrict__ scale, int T, int early_trigger) {
    constexpr int LG = G / 32;                        // lanes per group
    constexpr int L = LG == 2 ? 1 : LG == 4 ? 2 : 3;  // cross-lane stages
    static_assert(LG == 2 || LG == 4 || LG == 8, "group of 64, 128 or 256");
    extern __shared__ float red[];  // [blockDim.y][T / 32] warp maxima
    // Launched as a programmatic dependent, the kernel ahead of this one may
    // still be running: nothing is read or written before the wait.  The GEMM /
    // GEMV that consumes the codes reads only weight operands before its own
    // wait, so it may be let in before ours when the caller declared the
    // weights settled (early_trigger), else right after it.
    if (early_trigger) pdl_launch_dependents();
    pdl_wait();
    if (!early_trigger) pdl_launch_dependents();
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int q = lane & (LG - 1);
    const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.y + threadIdx.y;
    const bool row_ok = row < M;
    const int nunits = K >> 5;
    uint32_t qb[3];
    int cm;
    lane_map<L>(q, qb, cm);

    // load: register element e <- position e ^ cm (16- or 8-byte pieces).
    // Rows past M and units past K read row 0 / unit 0 instead: their values
    // never reach a stored code or the absmax of a stored row.
    uint32_t ra[U][16], rb[U][16];
#pragma unroll
    for (int j = 0; j < U; ++j) {
        const int u = t + j * T;
        const int64_t off = (row_ok ? row * ldx : 0) + (u < nunits ? static_cast<int64_t>(u) * 32 : 0);
        const __nv_bfloat16 *src = x + off;
        if constexpr (ACT == static_cast<int>(Act::kGluF32)) {
            // f32 input: 4-element pieces (cm has no bit below 4), elements
            // 0..15 into ra, 16..31 into rb
            const float *srcf = reinterpret_cast<const float *>(x) + off;
#pragma unroll
            for (int rc = 0; rc < 8; ++rc) {
                const int pc = rc ^ (cm >> 2);
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(srcf + 4 * pc));
                uint32_t *r = rc < 4 ? &ra[j][4 * rc] : &rb[j][4 * rc - 16];
                r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
            }
        } else if constexpr (L < 3) {
#pragma unroll
            for (int rc = 0; rc < 4; ++rc) {
                const int pc = rc ^ (cm >> 3);
                const uint4 va = __ldg(reinterpret_cast<const uint4 *>(src + 8 * pc));
                ra[j][4 * rc] = va.x; ra[j][4 * rc + 1] = va.y;
                ra[j][4 * rc + 2] = va.z; ra[j][4 * rc + 3] = va.w;
                if constexpr (ACT == static_cast<int>(Act::kSwiglu)) {
                    const uint4 vb = __ldg(reinterpret_cast<const uint4 *>(src + K + 8 * pc));
                    rb[j][4 * rc] = vb.x; rb[j][4 * rc + 1] = vb.y;
                    rb[j][4 * rc + 2] = vb.z; rb[j][4 * rc + 3] = vb.w;
                }
            }
        } else {
#pragma unroll
            for (int rh = 0; rh < 8; ++rh) {
                const int ph = rh ^ (cm >> 2);
                const uint2 va = __ldg(reinterpret_cast<const uint2 *>(src + 4 * ph));
                ra[j][2 * rh] = va.x; ra[j][2 * rh + 1] = va.y;
                if constexpr (ACT == static_cast<int>(Act::kSwiglu)) {
                    const uint2 vb = __ldg(reinterpret_cast<const uint2 *>(src + K + 4 * ph));
                    rb[j][2 * rh] = vb.x; rb[j][2 * rh + 1] = vb.y;
                }
            }
        }
    }
    float2 w[U][16];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < U; ++j) {
        rotate_unit<ACT, L>(ra[j], rb[j], qb, w[j]);
        if (t + j * T < nunits) amax = fmaxf(amax, unit_absmax(w[j]));
    }
    amax = team_absmax(amax, red, T >> 5, lane, t);
    constexpr float c = static_cast<float>(InvSqrtG<G>::v);
    const float s = __fdiv_rn(amax * c, 127.0f);  // max |f32(v / sqrt g)| / 127
    if (t == 0 && row_ok) scale[row] = s;
    if (!row_ok) return;
    const bool in_range = scale_in_range(amax);
    const float rs = __frcp_rn(s);
#pragma unroll
    for (int j = 0; j < U; ++j) {
        const int u = t + j * T;
        if (u >= nunits) continue;
        // element offset of unit row 0, position cm of this lane's group
        const int64_t base = row * K + static_cast<int64_t>(u - q) * 32 + cm;
        quantize_unit<G, OUT>(w[j], s, rs, in_range, qb, q16, q8, base);
    }
}

template <int ACT, int G, int U, int OUT>
cudaError_t launch_act(const void *x, int64_t M, int64_t K, int64_t ldx, int8_t *q8, void *q16,
                       float *scale, int T, int rows_per_cta, const LaunchCtx &ctx) {
    auto kern = rotate_quantize_act_kernel<ACT, G, U, OUT>;
    {
        // rows per CTA: the fewest waves of resident CTAs, ties to the default
        // (256 threads).  The CTAs are latency-bound, so a launch takes about
        // as many CTA lifetimes as it has waves: at 4096 x 4096, 9 CTAs of one
        // row per SM make 3.0 waves (10.4 us), 4 CTAs of two rows 3.4 (11.3 us)
        const int sms = sm_count();
        auto waves = [&](int rpc) -> int64_t {
            const int per_sm = resident_blocks_per_sm(reinterpret_cast<const void *>(kern), T * rpc,
                                                      sizeof(float) * static_cast<size_t>(rpc) * (T / 32));
            if (per_sm < 1 || sms < 1) return INT64_MAX;
            const int64_t slots = static_cast<int64_t>(per_sm) * sms;
            return ((M + rpc - 1) / rpc + slots - 1) / slots;
        };
        int64_t best = waves(rows_per_cta);
        const int dflt = rows_per_cta;
        for (int rpc = 1; rpc * T <= 512 && rpc <= 16; rpc *= 2) {
            if (rpc == dflt) continue;
            const int64_t w = waves(rpc);
            if (w < best) {
                best = w;
                rows_per_cta = rpc;
            }
        }
    }
    const dim3 block(T, rows_per_cta);
    const int64_t nsets = (M + rows_per_cta - 1) / rows_per_cta;
    const size_t smem = sizeof(float) * static_cast<size_t>(rows_per_cta) * (T / 32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nsets));
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ctx.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const __nv_bfloat16 *>(x), static_cast<int>(M),
                              static_cast<int>(K), ldx, q8, static_cast<__half *>(q16), scale, T,
                              ctx.early_trigger ? 1 : 0);
}

template <int ACT, int OUT>
cudaError_t dispatch_act(int g, int U, const void *x, int64_t M, int64_t K, int64_t ldx,
                         int8_t *q8, void *q16, float *scale, int T, int rpc,
                         const LaunchCtx &ctx) {
#define CK_ACT_CASE(GG)                                                                       \
    case GG:                                                                                  \
        return U == 1 ? launch_act<ACT, GG, 1, OUT>(x, M, K, ldx, q8, q16, scale, T, rpc, ctx) \
                      : launch_act<ACT, GG, 2, OUT>(x, M, K, ldx, q8, q16, scale, T, rpc, ctx);
    switch (g) {
        CK_ACT_CASE(64)
        CK_ACT_CASE(128)
        CK_ACT_CASE(256)
        default: return cudaErrorInvalidValue;
    }
#undef CK_ACT_CASE
}

template <typename TIn, typename TAcc, int ACT, int G, int U, int OUT>
cudaError_t launch_t(const void *x, int64_t M, int64_t K, int64_t ldx, int8_t *q8, void *q16,
                     float *scale, int T, int rows_per_cta, int qmax, const LaunchCtx &ctx) {
    const dim3 block(T, rows_per_cta);
    const size_t smem = 2 * sizeof(float) * static_cast<size_t>(rows_per_cta) * (T / 32);
    auto kern = rotate_quantize_kernel<TIn, TAcc, ACT, G, U, OUT>;
    // persistent-style grid: as many CTAs as fit at once (each walks rows)
    const int per_sm = resident_blocks_per_sm(reinterpret_cast<const void *>(kern), T * rows_per_cta, smem);
    const int resident = sm_count() * (per_sm > 0 ? per_sm : 1);
    if (resident < 1) return cudaErrorInvalidDevice;
    const int64_t groups = (M + rows_per_cta - 1) / rows_per_cta;
    const dim3 grid(static_cast<unsigned>(groups < resident ? groups : resident));
    kern<<<grid, block, smem, ctx.stream>>>(
        static_cast<const TIn *>(x), static_cast<int>(M), static_cast<int>(K), ldx, q8,
        static_cast<__half *>(q16), scale, T, qmax);
    return cudaGetLastError();
}

template <typename TIn, typename TAcc, int ACT, int G, int OUT>
cudaError_t dispatch_r(int U, const void *x, int64_t M, int64_t K, int64_t ldx, int8_t *q8,
                       void *q16, float *scale, int T, int rpc, int qmax, const LaunchCtx &ctx) {
    if (U == 1) return launch_t<TIn, TAcc, ACT, G, 1, OUT>(x, M, K, ldx, q8, q16, scale, T, rpc, qmax, ctx);
    return launch_t<TIn, TAcc, ACT, G, 2, OUT>(x, M, K, ldx, q8, q16, scale, T, rpc, qmax, ctx);
}

template <typename TIn, typename TAcc, int ACT, int OUT>
cudaError_t dispatch_g(int g, int R, const void *x, int64_t M, int64_t K, int64_t ldx,
                       int8_t *q8, void *q16, float *scale, int T, int rpc, int qmax,
                       const LaunchCtx &ctx) {
    switch (g) {
        case 64: return dispatch_r<TIn, TAcc, ACT, 64, OUT>(R, x, M, K, ldx, q8, q16, scale, T, rpc, qmax, ctx);
        case 128: return dispatch_r<TIn, TAcc, ACT, 128, OUT>(R, x, M, K, ldx, q8, q16, scale, T, rpc, qmax, ctx);
        case 256: return dispatch_r<TIn, TAcc, ACT, 256, OUT>(R, x, M, K, ldx, q8, q16, scale, T, rpc, qmax, ctx);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_rotate_quantize(const void *x, bool x_f32, Act act, int g, int64_t M,
                                   int64_t K, int64_t ldx, int8_t *q8, void *q16, float *scale,
                                   const LaunchCtx &ctx, bool f64_rotation, int qmax) {
    if (M <= 0) return cudaSuccess;
    if (K % 32 != 0) return cudaErrorInvalidValue;
    const int64_t nunits = K / 32;  // 32-element units
    const int R = nunits > 512 ? 2 : 1;  // units per thread (2 only beyond K = 16384)
    const int T = static_cast<int>(((nunits + R - 1) / R + 31) / 32 * 32);
    if (T > 512) return cudaErrorInvalidValue;
    const int rpc = T >= 256 ? 1 : 256 / T;
    const int out = (q8 ? kOutI8 : 0) | (q16 ? kOutF16 : 0);
    if (f64_rotation) {
        // offline weight quantization: int8 codes only, float64 rotation
        if (act != Act::kNone || out != kOutI8 || qmax < 1 || qmax > 127) return cudaErrorInvalidValue;
        if (x_f32)
            return dispatch_g<float, double, 0, kOutI8>(g, R, x, M, K, ldx, q8, q16, scale, T, rpc,
                                                        qmax, ctx);
        return dispatch_g<__nv_bfloat16, double, 0, kOutI8>(g, R, x, M, K, ldx, q8, q16, scale, T,
                                                            rpc, qmax, ctx);
    }
    if (x_f32 != (act == Act::kGluF32)) return cudaErrorInvalidValue;
    if (out != kOutI8 && out != kOutF16) return cudaErrorInvalidValue;
    const int rpc_act = T >= 256 ? 1 : 256 / T;
    if (act == Act::kGluF32)
        return out == kOutI8
                   ? dispatch_act<2, kOutI8>(g, R, x, M, K, ldx, q8, q16, scale, T, rpc_act, ctx)
                   : dispatch_act<2, kOutF16>(g, R, x, M, K, ldx, q8, q16, scale, T, rpc_act, ctx);
    if (act == Act::kNone)
        return out == kOutI8
                   ? dispatch_act<0, kOutI8>(g, R, x, M, K, ldx, q8, q16, scale, T, rpc_act, ctx)
                   : dispatch_act<0, kOutF16>(g, R, x, M, K, ldx, q8, q16, scale, T, rpc_act, ctx);
    return out == kOutI8
               ? dispatch_act<1, kOutI8>(g, R, x, M, K, ldx, q8, q16, scale, T, rpc_act, ctx)
               : dispatch_act<1, kOutF16>(g, R, x, M, K, ldx, q8, q16, scale, T, rpc_act, ctx);
    return cudaErrorInvalidValue;
}

}  // namespace ck
