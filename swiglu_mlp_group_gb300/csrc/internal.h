// internal.h -- launchers shared between the kernel translation units and the
// C-ABI layer (api.cu).  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ck {

// Input of the activation quantizer: bf16 x; bf16 [gate | up] (silu(gate) *
// up formed in f32); or that product already formed in f32 by the gate|up
// GEMM's epilogue (kGluF32: f32 [M, ldx], rotated exactly as kSwiglu's).
enum class Act : int { kNone = 0, kSwiglu = 1, kGluF32 = 2 };

// Output selection of the rotate+quantize code stores: INT8 [M, K] row-major,
// fp16 [M, K] row-major, or INT8 into the small-M GEMV's shared-memory
// activation fragments holding 1, 2, 4 or 8 tokens (element e of a row at byte
// 32 T (e / 32) + e % 32 past that row's base, T the tokens held).
enum QuantOut : int { kOutI8 = 1, kOutF16 = 2, kOutFrag1 = 4, kOutFrag2 = 8, kOutFrag8 = 16, kOutFrag4 = 32 };
constexpr int kOutFrag = kOutFrag1 | kOutFrag2 | kOutFrag4 | kOutFrag8;

struct LaunchCtx {
    cudaStream_t stream = nullptr;
    unsigned int *status = nullptr;  // device status word
    uint64_t timeout_ns = 2000000000ull;
    bool pdl = false;                // launch with programmatic stream serialization
    // the call's weight operands are settled (ck_set_launch_overlap): the
    // activation quantizer lets its dependent launch before its own wait, the
    // fused small-M GEMV reads its weights before its wait
    bool early_trigger = false;
};

// [swiglu ->] group rotation -> per-row absmax/127 -> RNE codes.
// x: bf16 (or f32 when x_f32) [M, ldx]; codes written as int8 to q8 and/or as
// fp16 values to q16 (both [M, K] row-major, may be null when not selected).
// f64_rotation: rotate in float64 and round once to f32 (offline weights;
// int8 output only), codes of at most qmax in magnitude (127; 31 and 7 for
// 6- and 4-bit weights).  Otherwise the rotation runs in f32 on bf16 input,
// or on f32 input with act kGluF32, and qmax is 127.
cudaError_t launch_rotate_quantize(const void *x, bool x_f32, Act act, int g, int64_t M,
                                   int64_t K, int64_t ldx, int8_t *q8, void *q16, float *scale,
                                   const LaunchCtx &ctx, bool f64_rotation = false, int qmax = 127);

// int8 codes -> fp16 values (exact), n elements, n % 16 == 0, 16-byte aligned.
cudaError_t launch_widen_codes(const int8_t *q, int64_t n, void *out16, cudaStream_t stream);
// The same for a [gate | up] weight of N = 2I rows of K codes, rows
// interleaved: out row 2j = row j, out row 2j + 1 = row I + j.
cudaError_t launch_widen_codes_glu(const int8_t *q, int64_t N, int64_t K, void *out16,
                                   cudaStream_t stream);

// Pack int8 [N, K] codes + f32 [N] scales into the GEMV-resident layout.
cudaError_t launch_pack_gemv(const int8_t *Wq, const float *sw, int64_t N, int64_t K, void *out,
                             cudaStream_t stream);
size_t gemv_packed_bytes(int64_t N, int64_t K);
// The same layout for 4- or 6-bit codes (W4A8 / W6A8).
cudaError_t launch_pack_gemv_lowbit(const int8_t *Wq, const float *sw, int64_t N, int64_t K,
                                    int bits, void *out, cudaStream_t stream);
size_t gemv_packed_lowbit_bytes(int64_t N, int64_t K, int bits);

// What a GEMM writes (out_kind): bf16 y (dequantized, + bias, + residual),
// the raw int32 sums, or the SwiGLU product of interleaved gate / up columns.
enum GemmOut : int { kOutBf16 = 0, kOutS32 = 1, kOutGlu = 2 };

// Exact-integer GEMM on fp16-held codes with fused dequantization:
//   kOutBf16: y bf16 [M, N] = bf16(acc * sx[m] * sw[n] + bias[n] + residual[m, n])
//             (bias, residual optional; residual may be y itself)
//   kOutS32 : acc int32 [M, N]
//   kOutGlu : B16 rows interleaved (row 2j = gate row j, 2j + 1 = up row j of a
//             [gate | up] weight of N = 2I rows; sw, bias in the [gate | up]
//             order); out f32 [M, I] = silu(f32(g)) * f32(u), g and u the bf16
//             values kOutBf16 would give (no residual)
// A16: fp16 [M, K], B16: fp16 [N, K], both row-major, K % 64 == 0.
cudaError_t launch_gemm_codes(const void *A16, const void *B16, int64_t M, int64_t N, int64_t K,
                              const float *sx, const float *sw, const void *bias,
                              const void *residual, void *out, int out_kind, const LaunchCtx &ctx);

// The tile code launch_gemm_codes uses for M x K -> N on a GPU of `sms` SMs
// (64 / 128 / 256: one-SM tile width; 512 / 448 / 2128: CTA pairs with 256- /
// 224- / 128-column tiles; 4512: K split between two pairs); the forced code
// when the test hook set one.
int gemm_tile_choice(int64_t M, int64_t N, int64_t K, int sms);

// The same GEMM on CTA pairs (256 x pair_n tiles over two SMs, tcgen05
// cta_group::2); pair_n is 256, 224 or 128.
cudaError_t launch_gemm_codes_pair(const void *A16, const void *B16, int64_t M, int64_t N,
                                   int64_t K, const float *sx, const float *sw, const void *bias,
                                   const void *residual, void *out, int out_kind, int pair_n,
                                   const LaunchCtx &ctx);

// The same GEMM with K split between the two CTA pairs of a 4-CTA cluster,
// one 256 x 256 tile per cluster, the halves' int32 sums added on chip
// (kOutBf16 and kOutS32 only; K / 64 >= 2).
cudaError_t launch_gemm_codes_splitk(const void *A16, const void *B16, int64_t M, int64_t N, int64_t K,
                                     const float *sx, const float *sw, const void *bias, const void *residual,
                                     void *out, int out_kind, const LaunchCtx &ctx);

// 4-CTA clusters of the split-K kernel the current device holds at once (0 on
// error).
int splitk_resident_clusters();

// Test hook: force the GEMM variant: 64, 128 or 256 (one-SM tile width), 512,
// 448 or 2128 (CTA pairs with 256 x 256, 256 x 224, 256 x 128 tiles), 4512
// (256 x 256 tiles, K split between two pairs; the kOutGlu output falls back
// to the automatic choice); anything else = auto.
void set_forced_gemm_bn(int bn);

// Small-M GEMV over a packed layout of wbits-bit weight codes (8: the INT8
// layout; 4 / 6: the W4A8 / W6A8 layouts): y bf16 [M, N] (+ bias, + residual,
// which may be y itself); xq INT8 [M, K] codes.  With acc_out (test hook)
// the exact int32 sums go to acc_out [M, N] instead (the engines' own
// sums: 2^(8-b) times the b-bit codes' ones); sx may then be null.
cudaError_t launch_gemv_packed(const int8_t *xq, const float *sx, int64_t M, int64_t K,
                               const void *Wpacked, int wbits, int64_t N, const void *bias,
                               const void *residual, void *y, const LaunchCtx &ctx,
                               int32_t *acc_out = nullptr);

// The same GEMV with the activation quantized inside each CTA (one launch):
// x bf16 [M, ldx] (act none / swiglu, group g), only where gemv_fusable(M, K)
// (M * round_up(K / 32, 32) <= 512, the activation fragments staged in
// shared memory).
bool gemv_fusable(int64_t M, int64_t K);
cudaError_t launch_gemv_fused(const void *x, int64_t ldx, Act act, int g, int64_t M, int64_t K,
                              const void *Wpacked, int wbits, int64_t N, const void *bias,
                              const void *residual, void *y, const LaunchCtx &ctx);
// one per weight code width (gemv_fused*.cu)
cudaError_t launch_gemv_fused_w8(const void *x, int64_t ldx, Act act, int g, int64_t M, int64_t K,
                                 const void *Wpacked, int64_t N, const void *bias,
                                 const void *residual, void *y, const LaunchCtx &ctx);
cudaError_t launch_gemv_fused_w6(const void *x, int64_t ldx, Act act, int g, int64_t M, int64_t K,
                                 const void *Wpacked, int64_t N, const void *bias,
                                 const void *residual, void *y, const LaunchCtx &ctx);
cudaError_t launch_gemv_fused_w4(const void *x, int64_t ldx, Act act, int g, int64_t M, int64_t K,
                                 const void *Wpacked, int64_t N, const void *bias,
                                 const void *residual, void *y, const LaunchCtx &ctx);

// Issue rate of tcgen05.mma kind::f16 128 x 256 x 16 from shared memory on
// every SM (TFLOP/s), timed on ctx.stream.
cudaError_t measure_tcgen05_f16_tflops(double *tflops, const LaunchCtx &ctx);

// Dense throughput of mma.sync m16n8k32 s8 (TOPS), timed on `stream`.
cudaError_t measure_int8_mma_tops(double *tops, int *sink, cudaStream_t stream);

// CK_OK when the current device is a GB300; also yields the device address of
// the status word every bounded wait reports to (defined in api.cu).
int device_ready_status(unsigned int **status);
// Time limit of device-side waits set by ck_set_wait_timeout_ns (api.cu).
uint64_t wait_timeout_ns();
// Whether ck_set_launch_overlap enabled overlapped launches (api.cu).
bool launch_overlap();

// A kernel that waits on a barrier nobody completes (timeout test hook).
cudaError_t launch_stalled_wait(const LaunchCtx &ctx);

}  // namespace ck
