/*
 * convrot_oracle.c -- plain, slow CPU oracle for the ConvRot INT8 W8A8 linear
 * and its fused SwiGLU variant.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code, no
 * header and no constant with the CUDA library in swiglu_mlp_group_gb300/;
 * the two are compared element by element on the same seeded inputs.
 *
 * Every step is written the way the method defines it, with no blocking,
 * fusion or reordering:
 *   - the rotation is an explicit float64 matrix product with an explicit
 *     Sylvester Hadamard matrix (no fast transform);
 *   - the quantizer divides (no reciprocal) and rounds half to even;
 *   - the GEMM is an int64 triple loop;
 *   - the dequantization is done in float64 and rounded once to f32, then to
 *     bf16 by this file's own bit-level round-to-nearest-even.
 * The only liberty taken is an OpenMP "parallel for" over independent output
 * rows, which leaves every result's arithmetic untouched.
 *
 * Sources (web pages; cited by title and section):
 *   [P1] sglang PR #44196, "comfy_kitchen SwiGLU MLP for Qwen-Image 2.1":
 *        Motivation; Accuracy Tests.
 *   [P3] sglang PR #35994 report, "Load serialized Comfy ConvRot INT8 DiTs":
 *        implementation breakdown (实现拆解); code excerpts (关键源码片段) of
 *        kitchen_int8.py and minimax_h3_weights.py; review notes (评论区精华).
 *   [P4] comfy-kitchen PR #277, "FP16 tensor-core fallback for int8_linear":
 *        The key observation; Notes for the reviewer.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <fenv.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Hadamard matrix.                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Sylvester construction H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]], in the
 * natural (Sylvester) order, scaled by 1/sqrt(g) so that H_g is orthogonal.
 * [P4] The key observation: the weight is stored as W_rot = W @ H^T and the
 * activation is rotated online, x_rot = x @ H.  [P3] kitchen_int8.py: the
 * rotation is parameterised by convrot_groupsize.
 * H is written row-major, g x g.  Returns 0, or -1 when g is not a power of two.
 */
ORACLE_API int oracle_sylvester_hadamard(int g, double *H) {
    if (g < 1 || (g & (g - 1)) != 0) return -1;
    /* unscaled +-1 entries first, built by doubling */
    H[0] = 1.0;
    for (int n = 1; n < g; n *= 2) {
        /* current block is n x n in the top-left corner of a g x g array */
        for (int i = 0; i < n; ++i) {
            for (int j = 0; j < n; ++j) {
                double h = H[(int64_t)i * g + j];
                H[(int64_t)i * g + (j + n)] = h;          /* top-right    =  H_n */
                H[(int64_t)(i + n) * g + j] = h;          /* bottom-left  =  H_n */
                H[(int64_t)(i + n) * g + (j + n)] = -h;   /* bottom-right = -H_n */
            }
        }
    }
    double s = 1.0 / sqrt((double)g);
    for (int64_t i = 0; i < (int64_t)g * g; ++i) H[i] *= s;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Group rotation.                                                           */
/* ------------------------------------------------------------------------ */

/*
 * Block-diagonal rotation of one row over contiguous groups of g along K:
 *   out[j*g + c] = sum_i v[j*g + i] * H_g[i, c]       (row vector times H_g)
 * in float64.  [P4] The key observation (x_rot = x @ H); [P3] kitchen_int8.py
 * create_weights (the rotated dimension must be divisible by the group size).
 */
static void rotate_one_row(const double *v, int64_t K, int g, const double *H, double *out) {
    for (int64_t j = 0; j < K / g; ++j) {
        for (int c = 0; c < g; ++c) {
            double acc = 0.0;
            for (int i = 0; i < g; ++i) acc += v[j * g + i] * H[(int64_t)i * g + c];
            out[j * g + c] = acc;
        }
    }
}

/*
 * Rotate `rows` rows of float64 input (row stride ldv elements) into out
 * [rows, K].  Returns 0, -1 for a g that is not a power of two, -2 when
 * K % g != 0, -3 on allocation failure.
 */
ORACLE_API int oracle_rotate_rows_f64(const double *v, int64_t rows, int64_t K, int64_t ldv,
                                      int g, double *out) {
    if (g < 1 || (g & (g - 1)) != 0) return -1;
    if (K % g != 0) return -2;
    double *H = (double *)malloc(sizeof(double) * (size_t)g * (size_t)g);
    if (!H) return -3;
    oracle_sylvester_hadamard(g, H);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) rotate_one_row(v + r * ldv, K, g, H, out + r * K);
    free(H);
    return 0;
}

/*
 * Same rotation for f32 input (row stride ldv): each row is widened exactly
 * to float64, rotated, and the result rounded once to f32.
 */
ORACLE_API int oracle_rotate_rows(const float *v, int64_t rows, int64_t K, int64_t ldv, int g,
                                  float *out) {
    if (g < 1 || (g & (g - 1)) != 0) return -1;
    if (K % g != 0) return -2;
    double *H = (double *)malloc(sizeof(double) * (size_t)g * (size_t)g);
    if (!H) return -3;
    oracle_sylvester_hadamard(g, H);
    int failed = 0;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double *vd = (double *)malloc(sizeof(double) * (size_t)K * 2);
        if (!vd) {
            failed = 1;
            continue;
        }
        double *od = vd + K;
        for (int64_t k = 0; k < K; ++k) vd[k] = (double)v[r * ldv + k];
        rotate_one_row(vd, K, g, H, od);
        for (int64_t k = 0; k < K; ++k) out[r * K + k] = (float)od[k];
        free(vd);
    }
    free(H);
    return failed ? -3 : 0;
}

/* ------------------------------------------------------------------------ */
/* Per-row absmax INT8 quantization.                                         */
/* ------------------------------------------------------------------------ */

/*
 * For each row: absmax = max_k |v[k]| (f32), scale = absmax / 127 (f32 IEEE
 * division), q[k] = clamp(round_half_even(v[k] / scale), -127, 127).  A row of
 * zeros gets scale 0 and codes 0.
 * [P3] kitchen_int8.py process_weights_after_loading: per_channel=True,
 * stochastic_rounding=0 (deterministic rounding), F32 scale per output row;
 * [P4] Notes for the reviewer: the activation is quantized per row on the same
 * INT8 grid as the weight.
 */
ORACLE_API void oracle_quantize_rows(const float *v, int64_t rows, int64_t K, int8_t *q,
                                     float *scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float *vr = v + r * K;
        float absmax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(vr[k]);
            if (a > absmax) absmax = a;
        }
        float s = absmax / 127.0f;
        scale[r] = s;
        for (int64_t k = 0; k < K; ++k) {
            float c;
            if (s == 0.0f) {
                c = 0.0f;
            } else {
                float t = vr[k] / s;
                c = nearbyintf(t); /* default FE_TONEAREST: ties to even */
                if (c > 127.0f) c = 127.0f;
                if (c < -127.0f) c = -127.0f;
            }
            q[r * K + k] = (int8_t)c;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* SwiGLU input activation.                                                  */
/* ------------------------------------------------------------------------ */

/*
 * a[r, j] = f32( silu(gate) * up ), gate = h[r, j], up = h[r, I + j], with
 * silu(z) = z / (1 + exp(-z)) evaluated in float64 and the product rounded
 * once to f32.  [P1] Motivation and Accuracy Tests: the down-projection's
 * quantizer applies silu(gate) * up in FP32 instead of rounding it to BF16,
 * and the packed weight is [gate | up] (gate first).
 * h is f32 with row stride ldh >= 2*I; a is [rows, I].
 */
ORACLE_API void oracle_swiglu(const float *h, int64_t rows, int64_t I, int64_t ldh, float *a) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < I; ++j) {
            double gt = (double)h[r * ldh + j];
            double up = (double)h[r * ldh + I + j];
            double silu = gt / (1.0 + exp(-gt));
            a[r * I + j] = (float)(silu * up);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* INT8 GEMM with wide integer accumulation.                                 */
/* ------------------------------------------------------------------------ */

/*
 * acc[m, n] = sum_k xq[m, k] * wq[n, k], accumulated in int64 (the int32 of
 * the method never overflows for K <= 133,000; int64 makes that a non-issue).
 * [P4] Summary and Measured results: INT8 x INT8 GEMM with int32 accumulation,
 * computed in the rotated basis, y = x_rot @ W_rot^T.
 */
ORACLE_API void oracle_int8_gemm(const int8_t *xq, const int8_t *wq, int64_t M, int64_t N,
                                 int64_t K, int64_t *acc) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)xq[m * K + k] * (int64_t)wq[n * K + k];
            acc[m * N + n] = s;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* f32 -> bf16, round to nearest even, bit level.                            */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/*
 * bf16 keeps the upper 16 bits of an f32.  Round to nearest, ties to even:
 * add 0x7FFF plus the lowest kept bit, then truncate.  NaN stays a (quiet)
 * NaN; overflow past the largest finite bf16 rounds to infinity as IEEE does.
 */
ORACLE_API uint16_t oracle_f32_to_bf16_bits(float f) {
    uint32_t u = f32_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN: keep sign, force quiet */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

ORACLE_API float oracle_bf16_bits_to_f32(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------------ */
/* Dequantization epilogue.                                                  */
/* ------------------------------------------------------------------------ */

/*
 * y[m, n] = bf16_rne( f32( acc[m,n] * sx[m] * sw[n] + bias[n] + res[m,n] ) ),
 * the product and sums in float64.  bias_bf16 [N] and res_bf16 [M, N] may be
 * NULL (no bias / no residual).  [P4] Summary / Changes: dequantize with the
 * per-token and per-output-row scales, bias/residual part of int8_linear's
 * contract; [P2] Commits and Description name a residual fused into the
 * linear without a formula: the residual is added in the epilogue, before the
 * one rounding to bf16.
 */
ORACLE_API void oracle_dequant(const int64_t *acc, const float *sx, const float *sw,
                               const uint16_t *bias_bf16, const uint16_t *res_bf16, int64_t M,
                               int64_t N, uint16_t *y) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double v = (double)acc[m * N + n] * (double)sx[m] * (double)sw[n];
            if (bias_bf16) v += (double)oracle_bf16_bits_to_f32(bias_bf16[n]);
            if (res_bf16) v += (double)oracle_bf16_bits_to_f32(res_bf16[m * N + n]);
            y[m * N + n] = oracle_f32_to_bf16_bits((float)v);
        }
    }
}

/* Element-wise f32 -> bf16 rounding of an array (used by the staged path). */
ORACLE_API void oracle_round_to_bf16(const float *in, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16_bits(in[i]);
}

/* ------------------------------------------------------------------------ */
/* GEMV-resident weight layout (codes and scales interleaved).               */
/* ------------------------------------------------------------------------ */

/*
 * The relayout that interleaves weights and their scales into one linear
 * stream for the small-M GEMV (comfy-kitchen PR #248, "Performance
 * improvements for qwen 3.x (Part 2)", Description: interleaving the weights
 * and their scales linearizes access; weight relayout kernels).  The page
 * does not fix the tiling; the one used here: for each 16-row tile t (rows
 * padded with zero codes and zero scales to a multiple of 16), K/32 blocks of
 * 512 bytes, then the tile's 16 f32 scales.  In block b, lane l (0..31) owns
 * bytes [16 l, 16 l + 16): with grp = l / 4, tg = l % 4, r = j / 4 and
 * i = j % 4, byte j holds the code at
 *   row = grp + 8 * (r % 2),
 *   col = 32 b + 8 * tg + 4 * (r / 2) + i
 * -- the A-operand fragment a0..a3 of one m16n8k32 INT8 tensor-core MMA (PTX
 * ISA, matrix fragments of mma.m16n8k32 for .s8, matrix A: a0 / a2 row
 * groupID, a1 / a3 row groupID + 8; a0, a1 hold k = 4 tg + i, a2, a3 hold
 * k = 16 + 4 tg + i) with k = 4 tg + i read from column 8 tg + i and
 * k = 16 + 4 tg + i from column 8 tg + 4 + i.
 * out must hold ceil(N / 16) * (K * 16 + 64) bytes; K % 32 == 0.
 */
ORACLE_API void oracle_pack_gemv(const int8_t *Wq, const float *sw, int64_t N, int64_t K,
                                 uint8_t *out) {
    const int64_t tiles = (N + 15) / 16;
    const int64_t nblk = K / 32;
    const int64_t tile_bytes = nblk * 512 + 64;
    for (int64_t t = 0; t < tiles; ++t) {
        uint8_t *tp = out + t * tile_bytes;
        for (int64_t b = 0; b < nblk; ++b) {
            for (int l = 0; l < 32; ++l) {
                const int grp = l / 4, tg = l % 4;
                for (int j = 0; j < 16; ++j) {
                    const int r = j / 4, i = j % 4;
                    const int row = grp + 8 * (r % 2);
                    const int64_t col = 32 * b + 8 * tg + 4 * (r / 2) + i;
                    const int64_t n = 16 * t + row;
                    const int8_t code = (n < N) ? Wq[n * K + col] : 0;
                    tp[b * 512 + 16 * l + j] = (uint8_t)code;
                }
            }
        }
        for (int r = 0; r < 16; ++r) {
            const int64_t n = 16 * t + r;
            const float s = (n < N) ? sw[n] : 0.0f;
            memcpy(tp + nblk * 512 + 4 * r, &s, 4);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Low-bit weights: W4A8 and W6A8.                                           */
/* ------------------------------------------------------------------------ */

/*
 * Per-row symmetric quantization to signed codes of at most qmax in
 * magnitude (qmax = 7 for 4-bit, 31 for 6-bit codes): absmax = max_k |v[k]|
 * (f32), scale = absmax / qmax (f32 IEEE division), q[k] = clamp(
 * round_half_even(v[k] / scale), -qmax, qmax); a row of zeros gets scale 0 and
 * codes 0.  The W4A8 / W6A8 weights of comfy-kitchen PR #248 ("Performance
 * improvements for qwen 3.x (Part 2)", Commits and Description) name the
 * formats without defining them; this is the reading that keeps every other
 * step of the ConvRot linear (the rotation, the per-row F32 scale, the INT8
 * activation, the exact integer sum and the dequantization) unchanged.
 */
ORACLE_API void oracle_quantize_rows_bits(const float *v, int64_t rows, int64_t K, int qmax,
                                          int8_t *q, float *scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float *vr = v + r * K;
        float absmax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(vr[k]);
            if (a > absmax) absmax = a;
        }
        float s = absmax / (float)qmax;
        scale[r] = s;
        for (int64_t k = 0; k < K; ++k) {
            float c;
            if (s == 0.0f) {
                c = 0.0f;
            } else {
                c = nearbyintf(vr[k] / s); /* ties to even */
                if (c > (float)qmax) c = (float)qmax;
                if (c < -(float)qmax) c = -(float)qmax;
            }
            q[r * K + k] = (int8_t)c;
        }
    }
}

/*
 * GEMV-resident layout of 4- or 6-bit codes.  Tiles, blocks and scales as in
 * oracle_pack_gemv; a block holds 32 * 2 * bits bytes (256 for 4-bit, 384
 * for 6-bit codes).  Lane l owns 2 * bits bytes, as 32-bit words: words 0
 * and 1 at bytes [8 l, 8 l + 8) of the block, and (6-bit only) word 2 at
 * bytes [256 + 4 l, 256 + 4 l + 4) -- so that each of the lane's loads is
 * one naturally aligned 8- or 4-byte access, adjacent to its neighbours'.
 * Let f[0..15] be the lane's 16 codes in the order of oracle_pack_gemv (byte
 * j of its 16 bytes), u = f & (2^bits - 1) their two's-complement bit fields,
 * and byte p of the lane the byte p % 4 of its word p / 4.
 *   4-bit: byte p (0..7) = u[8 (p/4) + p%4] | u[8 (p/4) + 4 + p%4] << 4:
 *          the low nibbles of bytes 0..3 hold f[0..3], their high nibbles
 *          f[4..7]; bytes 4..7 likewise f[8..11] and f[12..15].
 *   6-bit: byte 4 w + i (w = 0, 1, 2; i = 0..3) = u[4 w + i] << 2 |
 *          (u[12 + i] >> 2 w) & 3: bits 2..7 hold f[4 w + i], the low two
 *          bits one third of f[12 + i].
 * Placed in the top bits of an INT8 lane, a code c is the INT8 value
 * c * 2^(8 - bits) (the page's decode of such weights on the INT8 grid); the
 * scales stored are the codes' own (sw of oracle_quantize_rows_bits).
 * out must hold ceil(N / 16) * (K / 32 * 64 * bits + 64) bytes; K % 32 == 0.
 * Returns 0, or -1 for bits other than 4 and 6.
 */
ORACLE_API int oracle_pack_gemv_lowbit(const int8_t *Wq, const float *sw, int64_t N, int64_t K,
                                       int bits, uint8_t *out) {
    if (bits != 4 && bits != 6) return -1;
    const int64_t tiles = (N + 15) / 16;
    const int64_t nblk = K / 32;
    const int64_t block_bytes = 64 * bits;
    const int64_t tile_bytes = nblk * block_bytes + 64;
    const uint32_t mask = (1u << bits) - 1u;
    for (int64_t t = 0; t < tiles; ++t) {
        uint8_t *tp = out + t * tile_bytes;
        for (int64_t b = 0; b < nblk; ++b) {
            for (int l = 0; l < 32; ++l) {
                const int grp = l / 4, tg = l % 4;
                uint32_t u[16];
                for (int j = 0; j < 16; ++j) {
                    const int r = j / 4, i = j % 4;
                    const int row = grp + 8 * (r % 2);
                    const int64_t col = 32 * b + 8 * tg + 4 * (r / 2) + i;
                    const int64_t n = 16 * t + row;
                    const int8_t code = (n < N) ? Wq[n * K + col] : 0;
                    u[j] = (uint32_t)(uint8_t)code & mask;
                }
                /* the lane's byte p lives at word[p / 4] + p % 4 */
                uint8_t *word[3];
                word[0] = tp + b * block_bytes + 8 * l;
                word[1] = word[0] + 4;
                word[2] = tp + b * block_bytes + 256 + 4 * l;
                if (bits == 4) {
                    for (int p = 0; p < 8; ++p)
                        word[p / 4][p % 4] =
                            (uint8_t)(u[8 * (p / 4) + p % 4] | (u[8 * (p / 4) + 4 + p % 4] << 4));
                } else {
                    for (int w = 0; w < 3; ++w)
                        for (int i = 0; i < 4; ++i)
                            word[w][i] = (uint8_t)((u[4 * w + i] << 2) | ((u[12 + i] >> (2 * w)) & 3u));
                }
            }
        }
        for (int r = 0; r < 16; ++r) {
            const int64_t n = 16 * t + r;
            const float s = (n < N) ? sw[n] : 0.0f;
            memcpy(tp + nblk * block_bytes + 4 * r, &s, 4);
        }
    }
    return 0;
}

/* Number of OpenMP threads the oracle's parallel loops will use (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
ORACLE_API int oracle_num_threads(void) { return omp_get_max_threads(); }
ORACLE_API void oracle_set_num_threads(int n) { omp_set_num_threads(n); }
#else
ORACLE_API int oracle_num_threads(void) { return 1; }
ORACLE_API void oracle_set_num_threads(int n) { (void)n; }
#endif
