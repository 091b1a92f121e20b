/*
 * ck.h -- C ABI of the GB300 (sm_103a) ConvRot INT8 W8A8 linear library.
 *
 * The method (web pages, cited by title and section):
 *   [P1] sglang PR #44196, "comfy_kitchen SwiGLU MLP for Qwen-Image 2.1",
 *        Motivation / Modifications / Accuracy Tests;
 *   [P2] comfy-kitchen PR #248, "Performance improvements for qwen 3.x
 *        (Part 2)", Description;
 *   [P3] sglang PR #35994 report, "Load serialized Comfy ConvRot INT8 DiTs",
 *        implementation breakdown and code excerpts (kitchen_int8.py,
 *        minimax_h3_weights.py);
 *   [P4] comfy-kitchen PR #277, "FP16 tensor-core fallback for int8_linear",
 *        Summary / The key observation / Notes for the reviewer.
 *
 * A ConvRot linear computes y = x W^T in a rotated basis: the weight is
 * stored rotated, W_rot = W H (H block-diagonal, one normalised Sylvester
 * Hadamard H_g per contiguous group of g input features), quantized per
 * output row to INT8 with an F32 scale sw[n] = absmax/127; each activation row
 * is rotated online, x_rot = x H, and quantized per token on the same grid
 * (sx[m]); the INT8 GEMM accumulates exact int32 and the result is
 * dequantized, y[m,n] = bf16(acc[m,n] * sx[m] * sw[n] + bias[n]) [P4].
 * The inverse rotation is never applied.
 *
 * Residual: every entry point that writes y takes an optional residual, bf16
 * [M, N] row-major (row stride N) or NULL, added in f32 to the dequantized
 * value before its one rounding to bf16,
 *   y[m,n] = bf16(acc[m,n] * sx[m] * sw[n] + bias[n] + residual[m,n]),
 * the residual fused into the dequant epilogue [P2: Commits, Description --
 * a residual fusion is named among the decode fusions, with no formula].
 * residual may be y itself (an in-place add): each element is read before it
 * is written, by the same thread.
 *
 * Names against the call list of the hot path: ck_convrot_quantize_weight
 * writes the row-major layout (the GEMV packing is ck_prepare_weight);
 * ck_rotate_quantize_act; ck_int8_linear (act none / swiglu, bias,
 * residual); ck_swiglu_mlp; ck_int8_gemv_smallM (scales always inside the
 * packed weight, x with a leading dimension, a caller workspace for the codes
 * of the calls that quantize in a separate kernel).  The additions:
 * ck_prepare_weight and the weight-layout argument, the residual, and
 * ck_int8_gemm_dequant / ck_int8_gemv_dequant (several projections on one
 * quantized input), and the W6A8 / W4A8 decode weights
 * (ck_convrot_quantize_weight_bits, the _W6 / _W4 GEMV layouts,
 * ck_packed_gemv_smallM / ck_packed_gemv_dequant).
 *
 * Conventions for every entry point:
 *  - Matrices are row-major with the reduction dimension K contiguous; a
 *    leading dimension (ld*) is in elements.
 *  - Every pointer to tensor data is a DEVICE pointer owned by the caller.
 *    The library allocates no device memory: calls that need temporary
 *    device memory take a caller-owned workspace (size from
 *    ck_workspace_bytes).  The library keeps only a small host-side cache.
 *  - Every call is asynchronous on the given CUDA stream (NULL = legacy
 *    default stream); results are ready when the stream reaches that point.
 *  - Every call validates all arguments first and returns a ck_status.  On
 *    any validation error nothing is launched and no memory is touched.
 *    Nothing falls back silently to another path.
 *  - Launch failures are reported as CK_ERR_CUDA (cudaGetLastError after the
 *    launch).  Device-side pipeline waits are bounded in time; a wait that
 *    runs out makes the kernel finish early and records CK_ERR_TIMEOUT in a
 *    device status word, read (and cleared) by ck_poll_device_status.
 *  - Only devices of compute capability 10.3 (GB300) are accepted.
 */
#ifndef CK_H_
#define CK_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CK_API __attribute__((visibility("default")))
#else
#define CK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, spelled without including the CUDA headers. */
typedef struct CUstream_st *ck_stream_t;

typedef enum {
    CK_OK = 0,
    CK_ERR_NULL = 1,               /* a required pointer is NULL */
    CK_ERR_SHAPE = 2,              /* a size or leading dimension is out of range */
    CK_ERR_DTYPE = 3,              /* unsupported element type */
    CK_ERR_GROUP = 4,              /* g not in {64, 128, 256}, or K % g != 0 */
    CK_ERR_ALIGN = 5,              /* a pointer is not 16-byte aligned */
    CK_ERR_WORKSPACE = 6,          /* workspace NULL or smaller than required */
    CK_ERR_UNSUPPORTED_DEVICE = 7, /* current device is not compute capability 10.3 */
    CK_ERR_CUDA = 8,               /* a CUDA runtime call or launch failed */
    CK_ERR_TIMEOUT = 9,            /* a device-side wait ran out (ck_poll_device_status) */
    CK_ERR_INVALID = 10            /* an enum argument has an unknown value */
} ck_status;

typedef enum { CK_F32 = 0, CK_BF16 = 1 } ck_dtype;

/* Input activation applied by the activation quantizer before rotation. */
typedef enum {
    CK_ACT_NONE = 0,
    /* x holds [gate | up] (2K columns); the quantizer rotates
     * a = silu(gate) * up computed in f32, silu(z) = z / (1 + exp(-z)) [P1]. */
    CK_ACT_SWIGLU = 1
} ck_input_act;

/* Device layouts of a quantized weight. */
typedef enum {
    /* int8 [N, K] codes, row-major: the serialized checkpoint layout [P3]. */
    CK_WLAYOUT_ROWMAJOR_I8 = 0,
    /* GEMM-resident layout: the same int8 codes held as fp16 values (every
     * integer |q| <= 127 is exact in fp16), [N, K] row-major, 2 bytes per
     * code.  GB300's tensor cores multiply 16-bit operands; holding the codes
     * widened lets the GEMM stream both operands with TMA untouched. */
    CK_WLAYOUT_GEMM_F16 = 1,
    /* GEMV-resident layout for M <= 8: codes and row scales interleaved in
     * one linear stream per 16-row tile (see ck_prepare_weight) [P2]. */
    CK_WLAYOUT_GEMV_PACKED = 2,
    /* The same stream for the W6A8 / W4A8 decode weights [P2: Commits,
     * Description -- 4- and 6-bit weights decoded on the INT8 grid]: 6- or
     * 4-bit codes (from ck_convrot_quantize_weight_bits) packed 12 or 8 bytes
     * per 16 codes (see ck_prepare_weight).  Read by ck_packed_gemv_*. */
    CK_WLAYOUT_GEMV_PACKED_W6 = 3,
    CK_WLAYOUT_GEMV_PACKED_W4 = 4,
    /* GEMM-resident layout of a packed [gate | up] weight (2I rows) with its
     * gate and up rows interleaved -- row 2j = gate row j, row 2j + 1 = up row
     * j, fp16-held codes as CK_WLAYOUT_GEMM_F16 -- so that the gate|up GEMM's
     * epilogue holds gate j and up j together and forms silu(gate) * up
     * itself (ck_swiglu_mlp) [P1: Motivation]. */
    CK_WLAYOUT_GEMM_F16_GLU = 5
} ck_wlayout;

/* Operations whose workspace size ck_workspace_bytes reports. */
typedef enum {
    CK_OP_INT8_LINEAR = 0,  /* (M, K, N, wlayout) */
    CK_OP_SWIGLU_MLP = 1,   /* (M, H as K, I as N, wlayout) */
    CK_OP_GEMV_SMALLM = 2,  /* (M, K, N, -) */
    CK_OP_DEBUG_GEMM_S32 = 3 /* (M, K, N, -) */
} ck_op;

/* Human-readable name of a status code (static string). */
CK_API const char *ck_status_string(ck_status st);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
CK_API int ck_version(void);

/* CK_OK when the current CUDA device is compute capability 10.3. */
CK_API ck_status ck_device_check(void);

/*
 * Offline ConvRot weight quantization [P3: kitchen_int8.py
 * process_weights_after_loading -- per_channel=True, convrot=True,
 * convrot_groupsize=g, stochastic_rounding=0; weight_scale F32 [out, 1]].
 *   W   : [N, K] row-major, f32 or bf16 (wdt), device.
 *   Wq  : out, int8 [N, K] row-major codes of W_rot = W H, device.
 *   sw  : out, f32 [N] (the checkpoint's [N, 1]) = max_k |W_rot[n,k]| / 127.
 * codes = clamp(round_half_even(W_rot / sw), -127, 127); a zero row gets
 * sw = 0 and codes 0.  Errors: CK_ERR_NULL, CK_ERR_SHAPE (N < 1, K < 1,
 * K > 32768), CK_ERR_GROUP, CK_ERR_DTYPE, CK_ERR_ALIGN (W, Wq not 16-byte
 * aligned), CK_ERR_UNSUPPORTED_DEVICE, CK_ERR_CUDA.
 */
CK_API ck_status ck_convrot_quantize_weight(const void *W, ck_dtype wdt, int64_t N, int64_t K, int g,
                                     int8_t *Wq, float *sw, ck_stream_t stream);

/*
 * ck_convrot_quantize_weight to b-bit codes, bits = 8, 6 or 4 (the W8A8,
 * W6A8 and W4A8 weights) [P2: Commits, Description -- 4- and 6-bit weight
 * decode; the format is this library's reading]: with qmax = 2^(bits-1) - 1,
 * sw = max_k |W_rot[n,k]| / qmax (f32 division) and codes = clamp(
 * round_half_even(W_rot / sw), -qmax, qmax), held one per int8 in Wq.  bits =
 * 8 is ck_convrot_quantize_weight.  Same arguments and errors, plus
 * CK_ERR_INVALID (bits).
 */
CK_API ck_status ck_convrot_quantize_weight_bits(const void *W, ck_dtype wdt, int64_t N, int64_t K,
                                                 int g, int bits, int8_t *Wq, float *sw,
                                                 ck_stream_t stream);

/*
 * Online activation rotation + per-token INT8 quantization [P4: The key
 * observation (x_rot = x @ H); Notes for the reviewer (same INT8 grid as the
 * weight)], with the optional SwiGLU input activation [P1: Motivation].
 *   x   : bf16 [M, ldx] device; act NONE reads columns [0, K); act SWIGLU
 *         reads gate = columns [0, K) and up = columns [K, 2K).
 *   xq  : out, int8 [M, K] codes; sx : out, f32 [M] scales (absmax / 127).
 * Errors: CK_ERR_NULL, CK_ERR_SHAPE (M < 1, K < 1, K > 32768, ldx too small
 * or not a multiple of 8), CK_ERR_GROUP, CK_ERR_INVALID (act), CK_ERR_ALIGN,
 * CK_ERR_UNSUPPORTED_DEVICE, CK_ERR_CUDA.
 */
CK_API ck_status ck_rotate_quantize_act(const void *x, int64_t M, int64_t K, int64_t ldx,
                                 ck_input_act act, int g, int8_t *xq, float *sx,
                                 ck_stream_t stream);

/*
 * Same as ck_rotate_quantize_act, but the codes are written as fp16 values
 * (xq16 : fp16 [M, K]; every |q| <= 127 is exact in fp16), the operand
 * format of ck_int8_gemm_dequant.  Lets several linears that read the same
 * input (e.g. q, k and v projections) quantize it once.  Same errors.
 */
CK_API ck_status ck_rotate_quantize_act_f16(const void *x, int64_t M, int64_t K, int64_t ldx,
                                            ck_input_act act, int g, void *xq16, float *sx,
                                            ck_stream_t stream);

/*
 * INT8 GEMM + dequantization on already-quantized activations [P4: Summary]:
 *   y[m, n] = bf16( (sum_k xq16[m,k] * W[n,k]) * sx[m] * sw[n] + bias[n]
 *                   + residual[m,n] ),
 * accumulated exactly in int32.  xq16 : fp16-held codes [M, K] (from
 * ck_rotate_quantize_act_f16), sx f32 [M]; W : CK_WLAYOUT_GEMM_F16 [N, K];
 * sw f32 [N]; bias bf16 [N] or NULL; residual bf16 [M, N] or NULL (may be y);
 * y out bf16 [M, N].  K % 64 == 0,
 * N % 8 == 0.  Errors: CK_ERR_NULL, CK_ERR_SHAPE, CK_ERR_ALIGN,
 * CK_ERR_UNSUPPORTED_DEVICE, CK_ERR_CUDA.
 */
CK_API ck_status ck_int8_gemm_dequant(const void *xq16, const float *sx, int64_t M, int64_t K,
                                      const void *W, const float *sw, int64_t N,
                                      const void *bias, const void *residual, void *y,
                                      ck_stream_t stream);

/* Bytes a prepared weight of the given layout occupies (0 for a bad layout). */
CK_API size_t ck_prepared_weight_bytes(ck_wlayout layout, int64_t N, int64_t K);

/*
 * Re-lay a quantized weight (int8 [N, K] row-major codes + f32 [N] scales)
 * into a resident layout, once, ahead of the forward passes [P2: Description
 * -- weight relayout facilities; the resident decode-layout hook].
 *   CK_WLAYOUT_GEMM_F16     : out = fp16 [N, K] codes; sw is not used (the
 *                             GEMM takes the scales separately).
 *   CK_WLAYOUT_GEMM_F16_GLU : out = fp16 [N, K] codes of a [gate | up]
 *                             weight (N = 2I, even), out row 2j = Wq row j,
 *                             out row 2j + 1 = Wq row I + j; sw not used.
 *   CK_WLAYOUT_GEMV_PACKED  : out = for each 16-row tile t (rows padded with
 *                             zero codes to a multiple of 16): K/32 blocks of
 *                             512 bytes, block b holding the 16 x 32 codes
 *                             W[16t .. 16t+15, 32b .. 32b+31] in the order
 *                             the GEMV's INT8 tensor-core fragments read
 *                             them -- byte 16 l + j (l < 32, j < 16; g = l/4,
 *                             c = l%4, r = j/4, i = j%4) is
 *                             W[16t + g + 8 (r%2), 32b + 8c + 4 (r/2) + i] --
 *                             then the tile's 16 f32 scales (64 bytes).
 *                             Requires K % 32 == 0.
 *   CK_WLAYOUT_GEMV_PACKED_W6 / _W4 : the same tiles with 6- / 4-bit codes
 *                             (Wq must hold codes within +-31 / +-7, e.g. from
 *                             ck_convrot_quantize_weight_bits; others lose
 *                             their high bits).  A block is 384 / 256 bytes.
 *                             Lane l's 16 codes f[0..15] (f[j] = the INT8
 *                             layout's byte 16 l + j), as bit fields u[j] =
 *                             f[j] & (2^b - 1), fill 32-bit words: words 0 and
 *                             1 at block bytes [8 l, 8 l + 8), word 2 (6-bit)
 *                             at [256 + 4 l, 256 + 4 l + 4); the lane's byte p
 *                             is byte p % 4 of word p / 4.
 *                               4-bit: byte p = u[8 (p/4) + p%4] |
 *                                      u[8 (p/4) + 4 + p%4] << 4.
 *                               6-bit: byte 4 w + i (w < 3, i < 4) =
 *                                      u[4 w + i] << 2 | (u[12 + i] >> 2 w) & 3.
 *                             Masked into the top bits of a byte, a code c
 *                             reads as the INT8 value c * 2^(8 - b), so the
 *                             GEMV runs the INT8 arithmetic on them unchanged
 *                             and takes the factor out of the row scale.
 * out must hold ck_prepared_weight_bytes(layout, N, K) bytes, 16-byte aligned.
 * Errors: CK_ERR_NULL, CK_ERR_SHAPE, CK_ERR_INVALID (layout), CK_ERR_ALIGN,
 * CK_ERR_WORKSPACE (out_bytes too small), CK_ERR_UNSUPPORTED_DEVICE, CK_ERR_CUDA.
 */
CK_API ck_status ck_prepare_weight(const int8_t *Wq, const float *sw, int64_t N, int64_t K,
                            ck_wlayout layout, void *out, size_t out_bytes, ck_stream_t stream);

/* Workspace bytes an operation needs (0 when it needs none). */
CK_API size_t ck_workspace_bytes(ck_op op, int64_t M, int64_t K, int64_t N, ck_wlayout wlayout);

/*
 * ConvRot INT8 W8A8 linear [P4: Summary, The key observation; P1: Motivation
 * for act = SWIGLU (int8_linear(..., input_act="swiglu"))]:
 *   y[m, n] = bf16( acc[m, n] * sx[m] * sw[n] + bias[n] + residual[m, n] ),
 *   acc = sum_k xq[m, k] * Wq[n, k] (exact int32), (xq, sx) the per-token
 *   quantization of rot(x) (or of rot(silu(gate) * up) for act = SWIGLU).
 *   x      : bf16 [M, ldx] (columns as in ck_rotate_quantize_act).
 *   W      : quantized weight in layout wlayout (ROWMAJOR_I8 or GEMM_F16);
 *            ROWMAJOR_I8 is widened into the workspace on every call, so
 *            resident callers should prepare CK_WLAYOUT_GEMM_F16 once.
 *   sw     : f32 [N];  bias : bf16 [N] or NULL;  y : out, bf16 [M, N];
 *   residual : bf16 [M, N] or NULL, may be y (x may be y as well: the
 *            quantizer has read all of x before the GEMM writes).
 *   ws     : workspace of ck_workspace_bytes(CK_OP_INT8_LINEAR, M, K, N,
 *            wlayout) bytes (activation codes and scales live there).
 * Errors: CK_ERR_NULL, CK_ERR_SHAPE (N not a multiple of 8 among others),
 * CK_ERR_GROUP, CK_ERR_INVALID, CK_ERR_ALIGN, CK_ERR_WORKSPACE,
 * CK_ERR_UNSUPPORTED_DEVICE, CK_ERR_CUDA.
 */
CK_API ck_status ck_int8_linear(const void *x, int64_t M, int64_t K, int64_t ldx, ck_input_act act,
                         const void *W, ck_wlayout wlayout, const float *sw, int64_t N, int g,
                         const void *bias, const void *residual, void *y, void *ws,
                         size_t ws_bytes, ck_stream_t stream);

/* Size of the built-in device scratch of ck_int8_linear_noalloc (bytes). */
#define CK_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * ck_int8_linear without a caller workspace, for callers that cannot allocate
 * device memory: code running under a host that owns and pre-plans all device
 * memory (an inference engine's plugin or enqueue step, a memory-budgeted
 * runtime), or a plain C caller with no allocator, where a cudaMalloc would be
 * forbidden, could fail at run time, or would synchronize the device.  The
 * source pages have no counterpart; the arithmetic is exactly ck_int8_linear's.
 *
 * The temporaries (fp16-held activation codes [M, K] and f32 scales [M]) live
 * in one file-scope device array of CK_NOALLOC_SCRATCH_BYTES bytes that every
 * GPU which loads the library holds until the process exits.  The entry point
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *   - W must be in CK_WLAYOUT_GEMM_F16 (prepare it once with ck_prepare_weight).
 *   - Needs round_up(M*K*2, 256) + 4*M <= CK_NOALLOC_SCRATCH_BYTES, else
 *     returns CK_ERR_WORKSPACE before launching anything.
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture.
 *   - Every call shares the one array and leaves its contents behind; each
 *     call overwrites everything it reads, so nothing needs clearing.  Calls
 *     that overlap on the GPU (different streams, or different threads without
 *     ordering) race on the array: serialize them.
 * Other arguments, errors and results as ck_int8_linear.
 */
CK_API ck_status ck_int8_linear_noalloc(const void *x, int64_t M, int64_t K, int64_t ldx,
                                        ck_input_act act, const void *W16, const float *sw,
                                        int64_t N, int g, const void *bias,
                                        const void *residual, void *y, ck_stream_t stream);

/*
 * Fused SwiGLU MLP [P1: Motivation / Modifications]: one packed [gate | up]
 * linear, h = linear(x, Wgu) (bf16 [M, 2I]), then the down linear whose
 * quantizer applies silu(gate) * up in f32: y = linear_swiglu(h, Wd).
 *   x   : bf16 [M, H];  Wgu : [2I, H] (rows 0..I-1 gate, I..2I-1 up) in
 *         layout wlayout, sgu f32 [2I], bgu bf16 [2I] or NULL;
 *   Wd  : [H, I] in layout wlayout, sd f32 [H], bd bf16 [H] or NULL;
 *   wlayout CK_WLAYOUT_GEMM_F16_GLU: Wgu in that layout (sgu, bgu still in
 *         the [gate | up] order) and Wd in CK_WLAYOUT_GEMM_F16.  The gate|up
 *         GEMM's epilogue then writes a = silu(gate) * up in f32 [M, I] from
 *         the bf16 gate and up it dequantizes (in the bytes h takes
 *         otherwise), and the down linear's quantizer rotates and rounds a;
 *         y is bit-identical to the CK_WLAYOUT_GEMM_F16 call's;
 *   residual : bf16 [M, H] or NULL, added by the down linear's epilogue (the
 *         block's skip connection; may be x or y);
 *   y   : out, bf16 [M, H];
 *   ws  : ck_workspace_bytes(CK_OP_SWIGLU_MLP, M, H, I, wlayout) bytes,
 *         holding in order, each piece starting on a 256-byte boundary: the
 *         fp16-held codes of x [M, H], their f32 scales [M], h bf16 [M, 2I],
 *         the fp16-held codes of silu(gate) * up [M, I], their scales [M],
 *         and (ROWMAJOR_I8 only) the widened weight of the current linear
 *         (GEMM_F16_GLU: a f32 [M, I] in place of h).
 * Errors: as ck_int8_linear.
 */
CK_API ck_status ck_swiglu_mlp(const void *x, int64_t M, int64_t H, int64_t I, const void *Wgu,
                        const float *sgu, const void *bgu, const void *Wd, const float *sd,
                        const void *bd, const void *residual, ck_wlayout wlayout, int g,
                        void *y, void *ws, size_t ws_bytes, ck_stream_t stream);

/*
 * Small-M (1 <= M <= 8) decode GEMV over the GEMV-resident layout [P2:
 * Description -- M < 8 memory-bandwidth optimized GEMV, weights and scales
 * interleaved; the page uses tensor cores rather than dp4a, here the INT8
 * tensor-core MMA serves from 3 tokens (INT8 weights: 5) and dp4a below,
 * measured faster there].  Same arithmetic as ck_int8_linear.
 *   x       : bf16 [M, ldx] (act as in ck_rotate_quantize_act);
 *   Wpacked : CK_WLAYOUT_GEMV_PACKED weight of N x K (ck_prepare_weight);
 *   bias    : bf16 [N] or NULL;  residual : bf16 [M, N] or NULL (may be y);
 *   y       : out, bf16 [M, N];
 *   ws      : ck_workspace_bytes(CK_OP_GEMV_SMALLM, M, K, N, -) bytes (the
 *             activation codes; untouched where every CTA quantizes x itself,
 *             as the page describes, in one kernel: M = 1 with K <= 16384,
 *             and M = 2 with K <= 8192 under ck_set_launch_overlap(1)).
 * Errors: CK_ERR_NULL, CK_ERR_SHAPE (M > 8, K % 32, N % 8), CK_ERR_GROUP,
 * CK_ERR_INVALID, CK_ERR_ALIGN, CK_ERR_WORKSPACE, CK_ERR_UNSUPPORTED_DEVICE,
 * CK_ERR_CUDA.
 */
CK_API ck_status ck_int8_gemv_smallM(const void *x, int64_t M, int64_t K, int64_t ldx,
                              ck_input_act act, const void *Wpacked, int64_t N, int g,
                              const void *bias, const void *residual, void *y, void *ws,
                              size_t ws_bytes, ck_stream_t stream);

/*
 * Small-M GEMV + dequantization on already-quantized activations (the GEMV
 * counterpart of ck_int8_gemm_dequant, for decode steps where several
 * projections read the same input) [P2: Description; P4: Summary]:
 *   y[m, n] = bf16( (sum_k xq[m,k] * W[n,k]) * sx[m] * sw[n] + bias[n]
 *                   + residual[m,n] ).
 * xq : INT8 codes [M, K] (ck_rotate_quantize_act), sx f32 [M], 1 <= M <= 8;
 * Wpacked : CK_WLAYOUT_GEMV_PACKED weight of N x K (scales inside); bias bf16
 * [N] or NULL; residual bf16 [M, N] or NULL (may be y); y out bf16 [M, N].
 * K % 32 == 0, N % 8 == 0.  Errors:
 * CK_ERR_NULL, CK_ERR_SHAPE, CK_ERR_ALIGN, CK_ERR_UNSUPPORTED_DEVICE,
 * CK_ERR_CUDA.
 */
CK_API ck_status ck_int8_gemv_dequant(const int8_t *xq, const float *sx, int64_t M, int64_t K,
                                      const void *Wpacked, int64_t N, const void *bias,
                                      const void *residual, void *y, ck_stream_t stream);

/*
 * ck_int8_gemv_smallM / ck_int8_gemv_dequant over any GEMV-resident layout:
 * wlayout = CK_WLAYOUT_GEMV_PACKED (INT8 weights, the same calls as those),
 * CK_WLAYOUT_GEMV_PACKED_W6 or CK_WLAYOUT_GEMV_PACKED_W4 (the W6A8 / W4A8
 * decode weights [P2: Commits, Description]).  With b-bit codes c and their
 * scale sw,
 *   y[m, n] = bf16( (sum_k xq[m,k] * c[n,k]) * sx[m] * sw[n] + bias[n]
 *                   + residual[m,n] ),
 * the sum exact in int32 (it is formed as 2^(8-b) times that sum on the INT8
 * grid; the power of two leaves every rounding unchanged).  Same arguments
 * and errors as the INT8 calls, plus CK_ERR_INVALID (wlayout not a GEMV
 * layout).
 */
CK_API ck_status ck_packed_gemv_smallM(const void *x, int64_t M, int64_t K, int64_t ldx,
                                       ck_input_act act, const void *Wpacked, ck_wlayout wlayout,
                                       int64_t N, int g, const void *bias, const void *residual,
                                       void *y, void *ws, size_t ws_bytes, ck_stream_t stream);
CK_API ck_status ck_packed_gemv_dequant(const int8_t *xq, const float *sx, int64_t M, int64_t K,
                                        const void *Wpacked, ck_wlayout wlayout, int64_t N,
                                        const void *bias, const void *residual, void *y,
                                        ck_stream_t stream);

/*
 * Synchronizes `stream`, then reads and clears the device status word that
 * bounded device-side waits write.  Returns CK_OK, CK_ERR_TIMEOUT (a kernel
 * gave up waiting and finished early; its outputs are not valid) or
 * CK_ERR_CUDA (the synchronization itself failed).
 */
CK_API ck_status ck_poll_device_status(ck_stream_t stream);

/*
 * Time limit, in nanoseconds, of every device-side wait in kernels launched
 * after this call (default 2e9 ns).  0 restores the default.
 */
CK_API void ck_set_wait_timeout_ns(uint64_t ns);

/*
 * Overlapped launches across calls (default 0 = off; a launch-mode setting,
 * not an operation of the pages).  Each call's activation quantizer is always
 * a programmatic dependent of the kernel ahead of it on the stream: it waits
 * for that kernel before touching memory, so an earlier kernel's tail hides
 * its launch.  With on != 0, additionally:
 *   - the GEMM / GEMV behind a quantizer may start before the quantizer's own
 *     wait, and ck_int8_gemm_dequant / ck_int8_gemv_dequant start before the
 *     work ahead of them has finished;
 *   - such a kernel reads its weight operands at once (the prepared weight,
 *     its scales, the bias), and everything else only after its wait.
 * The caller guarantees that no work still in flight on the stream writes
 * those weight operands: prepare them, then synchronize, before their first
 * use in this mode.  Calls on CK_WLAYOUT_ROWMAJOR_I8 weights (widened into
 * the workspace by the call itself) keep their GEMM behind the quantizer's
 * wait.  Results are bit-identical in both modes.  Process-wide; takes effect
 * for calls made after it.
 */
CK_API void ck_set_launch_overlap(int on);

/*
 * Test hook: raw int32 accumulators of the GEMM engine used by
 * ck_int8_linear, acc[m, n] = sum_k xq[m, k] * Wq[n, k], for bit-exact
 * comparison (no counterpart on the pages; it exposes [P4]'s int32
 * accumulation).  xq int8 [M, K], Wq int8 [N, K], acc out int32 [M, N]
 * (N % 8 == 0), ws = ck_workspace_bytes(CK_OP_DEBUG_GEMM_S32, M, K, N, -).
 * K must be a multiple of 64.
 */
CK_API ck_status ck_debug_int8_gemm_s32(const int8_t *xq, const int8_t *Wq, int64_t M, int64_t N,
                                 int64_t K, int32_t *acc, void *ws, size_t ws_bytes,
                                 ck_stream_t stream);

/*
 * Test hook: force the output-tile width of the GEMM engine (64, 128 or 256
 * columns on one SM, 512, 448 or 2128 for 256 x 256, 256 x 224 or 256 x 128
 * tiles on CTA pairs, 4512 for 256 x 256 tiles with K split between the two
 * CTA pairs of a 4-CTA cluster -- the SwiGLU-epilogue output of
 * CK_WLAYOUT_GEMM_F16_GLU and K < 128 then take the automatic choice; any
 * other value restores the automatic choice, which picks the variant from the
 * SM count and the number of tiles).  Results never depend on it; tests use
 * it to cover every variant on small problems.
 */
CK_API void ck_debug_force_gemm_tile(int bn);

/*
 * Test hook: the small-M GEMV's exact int32 sums, acc[m, n] = sum_k xq[m,k] *
 * c[n,k], where c are the codes of a GEMV-resident weight (wlayout
 * CK_WLAYOUT_GEMV_PACKED / _W6 / _W4) as its engines see them on the INT8
 * grid (the INT8 codes; 4 / 16 times the 6- / 4-bit codes), instead of the
 * dequantized output.  xq INT8 [M, K], 1 <= M <= 8, K % 32 == 0, N % 8 ==
 * 0; acc int32 [M, N].  The kernel of ck_packed_gemv_dequant, compiled with
 * its final store writing the sums instead of the dequantized output (same
 * engines, tiling and launch).
 * Errors: CK_ERR_NULL, CK_ERR_INVALID (wlayout), CK_ERR_SHAPE, CK_ERR_ALIGN,
 * CK_ERR_UNSUPPORTED_DEVICE, CK_ERR_CUDA.
 */
CK_API ck_status ck_debug_gemv_s32(const int8_t *xq, int64_t M, int64_t K, const void *Wpacked,
                                   ck_wlayout wlayout, int64_t N, int32_t *acc,
                                   ck_stream_t stream);

/*
 * Test hook, host only (no device needed): the GEMM tile variant the engine
 * picks for an M x K -> N GEMM on a GPU of sms SMs, as a code of
 * ck_debug_force_gemm_tile (the forced code while one is set).  The choice:
 * K >= 6144 with at most sms / 4 tiles of 256 x 256 splits K between two CTA
 * pairs (4512; at launch also only when the device holds that many 4-CTA
 * clusters at once, else the rule below); K <= 1024 with at most 2 rounds
 * of 128 x 128 tiles takes one-SM 128 x 128 tiles; otherwise the variant with
 * the least (rounds of tiles x columns per SM / measured per-variant
 * throughput).  Returns 0 for M, N or K < 1 or sms < 2.
 */
CK_API int ck_debug_gemm_tile_choice(int64_t M, int64_t N, int64_t K, int sms);

/*
 * Test hook: how ck_int8_gemv_smallM quantizes the activation -- 1 = always
 * the quantizer kernel then the GEMV, 2 = inside every GEMV CTA wherever the
 * shape allows it (M * round_up(K/32, 32) <= 512, staged fragments of
 * M <= 2 tokens x K codes or 8 x K within 48 KB); any other
 * value restores the automatic choice.  Results never depend on it (the codes
 * are the same bit for bit); tests use it to cover both paths.
 */
CK_API void ck_debug_force_gemv_quantizer(int mode);

/*
 * Diagnostic: measures the dense throughput of the legacy INT8 tensor-core
 * instruction (mma.sync m16n8k32 s8 x s8 -> s32) on the current device, in
 * tera-operations per second, by timing a register-only kernel on `stream`
 * (synchronizes it).  sm_103a has no INT8 kind of tcgen05.mma, so this is the
 * INT8 tensor peak that "% of dense INT8 peak" figures are quoted against.
 * sink: a caller-owned device int the kernel may write (keeps its work alive).
 */
CK_API ck_status ck_measure_int8_mma_tops(double *tops, int *sink, ck_stream_t stream);

/*
 * Diagnostic: the issue rate of the tensor-core instruction the GEMMs use,
 * tcgen05.mma.cta_group::1.kind::f16 at 128 x 256 x 16, in TFLOP/s for the
 * whole device: one thread per SM issues 8192 of them back to back from
 * shared memory into two alternating TMEM accumulators (zero operands, no
 * TMA, no epilogue), timed on `stream` (synchronizes it).  The GEMMs' own
 * tensor peak, beside the cuBLAS-measured bf16 peak.  A timed-out final wait
 * is reported by ck_poll_device_status.
 */
CK_API ck_status ck_measure_tcgen05_f16_tflops(double *tflops, ck_stream_t stream);

/*
 * Test hook: launches one tiny kernel whose pipeline barrier is never
 * completed, so its bounded wait runs out after ck_set_wait_timeout_ns and
 * the kernel returns early.  ck_poll_device_status must then report
 * CK_ERR_TIMEOUT.  Exercises the timeout path without hanging the GPU.
 */
CK_API ck_status ck_debug_stalled_wait(ck_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CK_H_ */
