// quant_core.cuh -- device pieces of the activation rotate + quantize path,
// shared by the standalone quantizer (rotate_quantize.cu) and the small-M GEMV
// that quantizes its few activation rows itself (gemv_kernel.cuh), so that
// both produce the same codes bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.h"

namespace ck {
namespace qc {

constexpr unsigned kFull = 0xffffffffu;

// silu(z) * u in f32, silu(z) = z / (1 + e^-z), with e^-z = 2^(-z log2 e) from
// the hardware base-2 exponential and 1 / (1 + e^-z) from the hardware
// reciprocal (each within a few 2^-23 relative).  The large codes of a row come
// from large positive z, where e^-z is small and the product stays within ~2 ulp
// of the correctly rounded one; for very negative z, e^-z overflows to
// infinity and the product goes to zero, as the exact one does.  The product
// is rounded to f32 on its own (no contraction into the rotation's first
// butterfly): the rotation's input is the f32 product, wherever it is formed
// -- here, or in the gate|up GEMM's epilogue.
__device__ __forceinline__ float silu_mul(float z, float u) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(__fmul_rn(z, -1.4426950408889634f)));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__fadd_rn(1.0f, e)));
    return __fmul_rn(__fmul_rn(z, r), u);
}

// 1/sqrt(g), as a double (rounded to f32 where the rotation runs in f32)
template <int G>
struct InvSqrtG;
template <> struct InvSqrtG<64> { static constexpr double v = 0.125; };
template <> struct InvSqrtG<128> { static constexpr double v = 0.08838834764831845; };
template <> struct InvSqrtG<256> { static constexpr double v = 0.0625; };

// ---------------------------------------------------------------------------
// Activation path (bf16 input, f32 rotation), written for issue efficiency.
//
// Lane layout.  A group of g elements is Lg = g/32 lanes of one warp, lane q
// of the group starting with the unit (32 elements) at group offset 32 q.
// The cross-lane part of the transform (H_Lg over the Lg units, for every
// position inside a unit) runs as L = log2(Lg) half-exchange stages: in stage
// i the lanes q and q ^ 2^i swap half of their data through 32-bit shuffles,
// so that each of them then holds both operands of the butterflies of the
// half it kept and computes both outputs.  After the L stages lane q holds
// all Lg units of its group at the 32/Lg consecutive positions starting at
//     cm(q) = sum_i q_i 2^(4-i)      (q_i: bit i of q),
// which is what it quantizes and stores.  To make every exchange use the
// same register indices in every lane, the unit is loaded with position
// p = e ^ cm(q) in register element e; the in-lane butterflies whose stride
// is a bit of cm(q) then put the sum in the register of the upper position,
// which an fma with a per-lane sign (+-1, exact) takes care of.  In stage i
// the lane with q_i = 1 computes (mine - partner's) = -(lower - upper): the
// output of unit row r in lane q therefore carries the sign
// (-1)^popcount(r & q), folded into the quantization multiplier (rounding to
// nearest is odd-symmetric, |.| is sign-blind).
//
// Elements are kept as 16 f32 pairs per unit; every butterfly above stride 1
// is one packed add/sub/fma.f32x2 per two butterflies (each lane rounded like
// the scalar instruction); the stride-1 stage is fused into the bf16 unpack.
//
// Quantization: the scale s = f32(absmax / sqrt g) / 127 (IEEE division), as
// the reference arithmetic defines it; the codes are the rotated values times
// the reciprocal of the scale (divide or multiply by the reciprocal is left
// open by the method; the difference is at most one code at rounding ties).
// With f = f32(f32(1/sqrt g) * f32(1/s)) and the unit row's sign folded in,
// one packed fma per two codes, v * f + (2^23 + 0x6600), rounds v * f to the
// nearest integer (ties to even) in one rounding: the sum lies in
// [2^23, 2^24), where the ulp is 1, and leaves 0x6600 + code in the low 16
// bits -- the binary16 pattern of 1536 + code, from which one packed half
// subtraction gives the code (the low byte is the INT8 code).  v * f is
// within ~3 ulps of z / s, so a code differs from rint(z / s) only where
// z / s lies within a few ulps of a half-integer.  Rows whose absmax is
// zero, outside [2^-100, 2^100] or not finite take IEEE divisions for every
// code.
// ---------------------------------------------------------------------------
union F2 {
    float2 f;
    unsigned long long u;
};
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    F2 x{a}, y{b}, r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.u) : "l"(x.u), "l"(y.u));
    return r.f;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    F2 x{a}, y{b}, r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.u) : "l"(x.u), "l"(y.u));
    return r.f;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    F2 x{a}, y{b}, r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.u) : "l"(x.u), "l"(y.u));
    return r.f;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    F2 x{a}, y{b}, z{c}, r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.u) : "l"(x.u), "l"(y.u), "l"(z.u));
    return r.f;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// (x0, x1) -> (x0 + x1, x0 - x1): the stride-1 butterfly of one element pair.
__device__ __forceinline__ float2 bfly1(float x0, float x1) { return make_float2(x0 + x1, x0 - x1); }

// 2^23 + 0x6600 (bit pattern 0x4B006600) and the binary16 pair (1536, 1536).
constexpr float kRoundMagic = 8414720.0f;
constexpr uint32_t kHalf1536x2 = 0x66006600u;

// fp16 code pair from two magic sums
__device__ __forceinline__ uint32_t codes_f16x2(float2 y) {
    const uint32_t h = prmt(__float_as_uint(y.x), __float_as_uint(y.y), 0x5410u);
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(h), "r"(kHalf1536x2));
    return d;
}
// four INT8 codes (low bytes of the magic sums), in element order
__device__ __forceinline__ uint32_t codes_i8x4(float2 y0, float2 y1) {
    const uint32_t lo = prmt(__float_as_uint(y0.x), __float_as_uint(y0.y), 0x0040u);
    const uint32_t hi = prmt(__float_as_uint(y1.x), __float_as_uint(y1.y), 0x0040u);
    return prmt(lo, hi, 0x5410u);
}

// Store the KS code pairs of one unit row: fp16 (4 KS bytes) or INT8 (2 KS bytes).
template <int KS, int OUT>
__device__ __forceinline__ void store_codes(const float2 (&y)[KS], __half *q16, int8_t *q8,
                                            int64_t off) {
    if constexpr ((OUT & kOutF16) != 0) {
        uint32_t h[KS];
#pragma unroll
        for (int k = 0; k < KS; ++k) h[k] = codes_f16x2(y[k]);
        if constexpr (KS >= 4) {
            uint4 *dst = reinterpret_cast<uint4 *>(q16 + off);
#pragma unroll
            for (int c = 0; c < KS / 4; ++c)
                dst[c] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
        } else {
            *reinterpret_cast<uint2 *>(q16 + off) = make_uint2(h[0], h[1]);
        }
    }
    if constexpr ((OUT & (kOutI8 | kOutFrag)) != 0) {
        uint32_t b[KS / 2];
#pragma unroll
        for (int k = 0; k < KS / 2; ++k) b[k] = codes_i8x4(y[2 * k], y[2 * k + 1]);
        // fragment layout: the 2 KS codes (aligned to their width) stay within
        // one 32-element block, at byte 32 T (e / 32) + e % 32
        constexpr int64_t kBlockBytes = (OUT & kOutFrag1)   ? 32
                                        : (OUT & kOutFrag2) ? 64
                                        : (OUT & kOutFrag4) ? 128
                                                            : 256;
        int8_t *dst = (OUT & kOutFrag) != 0 ? q8 + (off >> 5) * kBlockBytes + (off & 31) : q8 + off;
        if constexpr (KS == 8) {
            *reinterpret_cast<uint4 *>(dst) = make_uint4(b[0], b[1], b[2], b[3]);
        } else if constexpr (KS == 4) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(b[0], b[1]);
        } else {
            *reinterpret_cast<uint32_t *>(dst) = b[0];
        }
    }
}

// x0 + x1 and x0 - x1 for the bf16 pair (x0 low, x1 high) of one word, each
// rounded once to f32 (mixed-precision add/sub: a bf16 operand, an f32 one).
__device__ __forceinline__ float2 bfly1_bf16x2(uint32_t word) {
    const float x1 = __uint_as_float(word & 0xffff0000u);
    float2 r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %3;\n\t"
        "sub.rn.f32.bf16 %1, lo, %3;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(word), "f"(x1));
    return r;
}
// +-1.0f or +-v with the sign bit flipped where flip has bit 31 set
__device__ __forceinline__ float flip_sign(float v, uint32_t flip) {
    return __uint_as_float(__float_as_uint(v) ^ flip);
}

// ---- pieces of the activation kernel

// qb[i]: bit i of the lane's index q within its group, moved to bit 31
template <int L>
__device__ __forceinline__ void lane_map(int q, uint32_t (&qb)[3], int &cm) {
#pragma unroll
    for (int i = 0; i < 3; ++i) qb[i] = (static_cast<uint32_t>(q) >> i & 1u) << 31;
    cm = 0;
#pragma unroll
    for (int i = 0; i < L; ++i) cm |= ((q >> i) & 1) << (4 - i);
}

// One 32-element unit: unpack (+ swiglu), the in-lane butterflies and the
// cross-lane half-exchange stages.  Warp-collective (shuffles).  ra / rb:
// bf16 pairs of x (act none), of gate / up (act swiglu), or the f32 bits of
// register elements 0..15 / 16..31 (act kGluF32: the f32 product of swiglu,
// entering the butterflies exactly as swiglu's own product does).
template <int ACT, int L>
__device__ __forceinline__ void rotate_unit(const uint32_t (&ra)[16], const uint32_t (&rb)[16],
                                            const uint32_t (&qb)[3], float2 (&w)[16]) {
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        if constexpr (ACT == static_cast<int>(Act::kGluF32)) {
            const float x0 = __uint_as_float(m < 8 ? ra[2 * m] : rb[2 * m - 16]);
            const float x1 = __uint_as_float(m < 8 ? ra[2 * m + 1] : rb[2 * m - 15]);
            w[m] = bfly1(x0, x1);
        } else if constexpr (ACT == static_cast<int>(Act::kSwiglu)) {
            const float x0 = silu_mul(__uint_as_float(ra[m] << 16), __uint_as_float(rb[m] << 16));
            const float x1 = silu_mul(__uint_as_float(ra[m] & 0xffff0000u),
                                      __uint_as_float(rb[m] & 0xffff0000u));
            w[m] = bfly1(x0, x1);
        } else {
            w[m] = bfly1_bf16x2(ra[m]);
        }
    }
    // in-lane strides 2, 4, 8, 16 (pair strides 1, 2, 4, 8)
#pragma unroll
    for (int hs = 1; hs < 16; hs <<= 1) {
        const int s = 2 * hs;                 // element stride
        const bool may_swap = s >= (32 >> L);  // s is a bit of some lane's cm
        // stride 16 <-> q bit 0, 8 <-> bit 1, 4 <-> bit 2
        const uint32_t fl = may_swap ? qb[s == 16 ? 0 : s == 8 ? 1 : 2] : 0u;
        const float sg = flip_sign(1.0f, fl), nsg = flip_sign(-1.0f, fl);
        const float2 sg2 = make_float2(sg, sg), nsg2 = make_float2(nsg, nsg);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & hs) == 0) {
                const float2 p = w[i], r = w[i + hs];
                if (may_swap) {
                    w[i] = fma2(sg2, p, r);
                    w[i + hs] = fma2(nsg2, r, p);
                } else {
                    w[i] = add2(p, r);
                    w[i + hs] = sub2(p, r);
                }
            }
        }
    }
    // cross-lane half-exchange stages (unit strides 1 .. Lg/2)
#pragma unroll
    for (int i = 0; i < L; ++i) {
        const int KI = 16 >> i;  // pairs per unit row before this stage
        const int NR = 1 << i;   // unit rows held before this stage
        float2 nv[16];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
#pragma unroll
            for (int k = 0; k < KI / 2; ++k) {
                const float2 keep = w[r * KI + k], send = w[r * KI + KI / 2 + k];
                const float2 got = make_float2(__shfl_xor_sync(kFull, send.x, 1 << i),
                                               __shfl_xor_sync(kFull, send.y, 1 << i));
                nv[r * (KI / 2) + k] = add2(keep, got);
                nv[(r + NR) * (KI / 2) + k] = sub2(keep, got);
            }
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) w[m] = nv[m];
    }
}

// max(|a|, |b|, |c|) in one instruction (the three-input max with |.| on its inputs)
__device__ __forceinline__ float max3_abs(float a, float b, float c) {
    float d;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// max |w| over the unit
__device__ __forceinline__ float unit_absmax(const float2 (&w)[16]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = max3_abs(m, w[i].x, w[i].y);
    return m;
}

// Codes of one unit's worth of this lane's group (Lg unit rows x 2 KS
// positions starting at `base`), given s = row scale and rs = 1/s rounded.
template <int G, int OUT>
__device__ __forceinline__ void quantize_unit(const float2 (&w)[16], float s, float rs,
                                              bool in_range, const uint32_t (&qb)[3],
                                              __half *q16, int8_t *q8, int64_t base) {
    constexpr int LG = G / 32;
    constexpr int L = LG == 2 ? 1 : LG == 4 ? 2 : 3;
    constexpr int KS = 16 >> L;
    constexpr float c = static_cast<float>(InvSqrtG<G>::v);
    const float2 magic2 = make_float2(kRoundMagic, kRoundMagic);
    // c with the sign of unit row r: (-1)^popcount(r & q)
    auto crow = [&](int r) {
        uint32_t fl = 0;
#pragma unroll
        for (int i = 0; i < L; ++i)
            if (r >> i & 1) fl ^= qb[i];
        return flip_sign(c, fl);
    };
    if (in_range) {
        const float f = c * rs;  // 1 / (sqrt g s)
        uint32_t fl[LG];
#pragma unroll
        for (int r = 0; r < LG; ++r) fl[r] = __float_as_uint(crow(r)) & 0x80000000u;
#pragma unroll
        for (int r = 0; r < LG; ++r) {
            const float fr = flip_sign(f, fl[r]);
            const float2 f2 = make_float2(fr, fr);
            float2 y[KS];
#pragma unroll
            for (int k = 0; k < KS; ++k) y[k] = fma2(w[r * KS + k], f2, magic2);  // rint(v f)
            store_codes<KS, OUT>(y, q16, q8, base + 32 * r);
        }
    } else {
        // zero, subnormal-range or non-finite absmax: IEEE divisions throughout
#pragma unroll
        for (int r = 0; r < LG; ++r) {
            const float cr = crow(r);
            float2 y[KS];
#pragma unroll
            for (int k = 0; k < KS; ++k) {
                const float z0 = w[r * KS + k].x * cr, z1 = w[r * KS + k].y * cr;
                float a0 = s == 0.0f ? 0.0f : rintf(__fdiv_rn(z0, s));
                float a1 = s == 0.0f ? 0.0f : rintf(__fdiv_rn(z1, s));
                a0 = fminf(fmaxf(a0, -127.0f), 127.0f);
                a1 = fminf(fmaxf(a1, -127.0f), 127.0f);
                y[k] = make_float2(a0 + kRoundMagic, a1 + kRoundMagic);
            }
            store_codes<KS, OUT>(y, q16, q8, base + 32 * r);
        }
    }
}

// Row scale from the team's warp maxima: every thread reads them all.
__device__ __forceinline__ float team_absmax(float amax, float *red, int nw, int lane, int t) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
    if (lane == 0) red[threadIdx.y * nw + (t >> 5)] = amax;
    __syncthreads();
    amax = 0.0f;
    for (int ww = 0; ww < nw; ++ww) amax = fmaxf(amax, red[threadIdx.y * nw + ww]);
    return amax;
}
__device__ __forceinline__ bool scale_in_range(float amax) {
    return amax >= 0x1p-100f && amax <= 0x1p+100f;
}

}  // namespace qc
}  // namespace ck
