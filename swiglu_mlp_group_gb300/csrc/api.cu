// api.cu -- the C ABI declared in include/ck.h: argument validation,
// workspace carving and kernel sequencing.  Every entry point validates all
// of its arguments before it launches anything, and returns a ck_status.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "ck.h"
#include "internal.h"
#include "trace.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxK = 32768;
constexpr int64_t kMaxRows = (int64_t{1} << 31) - 1;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

// Device status word written by bounded device-side waits.
__device__ unsigned int g_device_status = 0;

std::mutex g_mu;
unsigned int *g_status_ptr[kMaxDevices] = {};
signed char g_device_ok[kMaxDevices] = {};  // 0 unknown, 1 ok, -1 unsupported
std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<bool> g_overlap{false};  // ck_set_launch_overlap
std::atomic<int> g_gemv_quant_mode{0};  // ck_debug_force_gemv_quantizer

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

// CK_OK when the current device is compute capability 10.3; also resolves the
// device address of the status word for that device.
ck_status device_ready(unsigned int **status) {
    const int dev = current_device();
    if (dev < 0) {
        cudaGetLastError();
        return CK_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_device_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return CK_ERR_UNSUPPORTED_DEVICE;
        }
        g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_device_ok[dev] != 1) return CK_ERR_UNSUPPORTED_DEVICE;
    if (g_status_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return CK_ERR_CUDA;
        }
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
    }
    if (status) *status = g_status_ptr[dev];
    return CK_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_group(int g) { return g == 64 || g == 128 || g == 256; }

// weight code width of a GEMV-resident layout (0: not one)
int gemv_layout_bits(int layout) {
    switch (layout) {
        case CK_WLAYOUT_GEMV_PACKED: return 8;
        case CK_WLAYOUT_GEMV_PACKED_W6: return 6;
        case CK_WLAYOUT_GEMV_PACKED_W4: return 4;
        default: return 0;
    }
}
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

ck_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CK_OK : CK_ERR_CUDA; }

ck::LaunchCtx make_ctx(ck_stream_t stream, unsigned int *status, bool pdl) {
    ck::LaunchCtx c;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    c.status = status;
    c.timeout_ns = g_timeout_ns.load();
    c.pdl = pdl;
    return c;
}

// The activation quantizer heading a call: always a programmatic dependent of
// the kernel ahead of it (it waits before touching memory); it lets the GEMM /
// GEMV behind it in before its own wait only when the caller declared the
// weights settled and the call reads them from where they rest.
ck::LaunchCtx quant_ctx(ck_stream_t stream, unsigned int *status, bool resident_weights) {
    ck::LaunchCtx c = make_ctx(stream, status, true);
    c.early_trigger = resident_weights && g_overlap.load();
    return c;
}

// Small-M GEMV: where the activation is quantized inside the GEMV's CTAs by
// default (measured on GB300 against the quantizer kernel + GEMV pair, 40
// calls back to back: M = 1 0.4-1.7 us faster; M = 2 0.5 us faster with
// overlapped launches, 0.5 us slower without; M = 4 0.1-1.5 us slower).
bool gemv_fuse_by_default(int64_t M, int64_t K) {
    return K > 0 && (M == 1 || (M == 2 && g_overlap.load()));
}

// Workspace plans ------------------------------------------------------------
struct LinearWs {
    size_t xq, sx, w16, total;
};
LinearWs linear_ws(int64_t M, int64_t K, int64_t N, ck_wlayout wl) {
    LinearWs w{};
    size_t off = 0;
    w.xq = off;
    off = round_up(off + static_cast<size_t>(M) * K * 2, 256);
    w.sx = off;
    off = round_up(off + static_cast<size_t>(M) * 4, 256);
    w.w16 = off;
    if (wl == CK_WLAYOUT_ROWMAJOR_I8) off = round_up(off + static_cast<size_t>(N) * K * 2, 256);
    w.total = off;
    return w;
}

struct MlpWs {
    size_t xq, sx, h, aq, sa, w16, total;
};
MlpWs mlp_ws(int64_t M, int64_t H, int64_t I, ck_wlayout wl) {
    MlpWs w{};
    size_t off = 0;
    w.xq = off;
    off = round_up(off + static_cast<size_t>(M) * H * 2, 256);
    w.sx = off;
    off = round_up(off + static_cast<size_t>(M) * 4, 256);
    w.h = off;
    off = round_up(off + static_cast<size_t>(M) * 2 * I * 2, 256);
    w.aq = off;
    off = round_up(off + static_cast<size_t>(M) * I * 2, 256);
    w.sa = off;
    off = round_up(off + static_cast<size_t>(M) * 4, 256);
    w.w16 = off;
    if (wl == CK_WLAYOUT_ROWMAJOR_I8) off = round_up(off + static_cast<size_t>(2 * I) * H * 2, 256);
    w.total = off;
    return w;
}

struct DebugWs {
    size_t a16, b16, total;
};
DebugWs debug_ws(int64_t M, int64_t K, int64_t N) {
    DebugWs w{};
    w.a16 = 0;
    w.b16 = round_up(static_cast<size_t>(M) * K * 2, 256);
    w.total = round_up(w.b16 + static_cast<size_t>(N) * K * 2, 256);
    return w;
}

template <typename T>
T *at(void *base, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(base) + off);
}

// Shared checks of a linear call (everything but the pointers' presence).
ck_status check_linear_shape(int64_t M, int64_t K, int64_t ldx, ck_input_act act, int64_t N,
                             int g) {
    if (act != CK_ACT_NONE && act != CK_ACT_SWIGLU) return CK_ERR_INVALID;
    if (M < 1 || K < 1 || N < 1 || M > kMaxRows || N > kMaxRows || K > kMaxK) return CK_ERR_SHAPE;
    const int64_t need = act == CK_ACT_SWIGLU ? 2 * K : K;
    if (ldx < need || ldx % 8 != 0) return CK_ERR_SHAPE;
    if (N % 8 != 0) return CK_ERR_SHAPE;
    if (!valid_group(g) || K % g != 0) return CK_ERR_GROUP;
    return CK_OK;
}

}  // namespace

namespace ck {
int device_ready_status(unsigned int **status) { return static_cast<int>(device_ready(status)); }
uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }
bool launch_overlap() { return g_overlap.load(); }
}  // namespace ck

extern "C" {

CK_API const char *ck_status_string(ck_status st) {
    switch (st) {
        case CK_OK: return "CK_OK";
        case CK_ERR_NULL: return "CK_ERR_NULL: a required pointer is NULL";
        case CK_ERR_SHAPE: return "CK_ERR_SHAPE: a size or leading dimension is out of range";
        case CK_ERR_DTYPE: return "CK_ERR_DTYPE: unsupported element type";
        case CK_ERR_GROUP: return "CK_ERR_GROUP: group size not in {64,128,256} or K % g != 0";
        case CK_ERR_ALIGN: return "CK_ERR_ALIGN: a pointer is not 16-byte aligned";
        case CK_ERR_WORKSPACE: return "CK_ERR_WORKSPACE: workspace missing or too small";
        case CK_ERR_UNSUPPORTED_DEVICE:
            return "CK_ERR_UNSUPPORTED_DEVICE: current device is not compute capability 10.3";
        case CK_ERR_CUDA: return "CK_ERR_CUDA: a CUDA call or kernel launch failed";
        case CK_ERR_TIMEOUT: return "CK_ERR_TIMEOUT: a device-side wait ran out";
        case CK_ERR_INVALID: return "CK_ERR_INVALID: unknown enum value";
    }
    return "unknown ck_status";
}

CK_API int ck_version(void) { return 205; }

CK_API ck_status ck_device_check(void) { return device_ready(nullptr); }

CK_API void ck_set_wait_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns == 0 ? kDefaultTimeoutNs : ns);
}

CK_API void ck_set_launch_overlap(int on) { g_overlap.store(on != 0); }

CK_API ck_status ck_convrot_quantize_weight(const void *W, ck_dtype wdt, int64_t N, int64_t K,
                                            int g, int8_t *Wq, float *sw, ck_stream_t stream) {
    CK_TRACE("ck_convrot_quantize_weight");
    return ck_convrot_quantize_weight_bits(W, wdt, N, K, g, 8, Wq, sw, stream);
}

CK_API ck_status ck_convrot_quantize_weight_bits(const void *W, ck_dtype wdt, int64_t N, int64_t K,
                                                 int g, int bits, int8_t *Wq, float *sw,
                                                 ck_stream_t stream) {
    CK_TRACE("ck_convrot_quantize_weight_bits");
    if (!W || !Wq || !sw) return CK_ERR_NULL;
    if (bits != 8 && bits != 6 && bits != 4) return CK_ERR_INVALID;
    if (wdt != CK_F32 && wdt != CK_BF16) return CK_ERR_DTYPE;
    if (N < 1 || K < 1 || N > kMaxRows || K > kMaxK) return CK_ERR_SHAPE;
    if (!valid_group(g) || K % g != 0) return CK_ERR_GROUP;
    if (!aligned16(W) || !aligned16(Wq)) return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    return from_cuda(ck::launch_rotate_quantize(W, wdt == CK_F32, ck::Act::kNone, g, N, K, K, Wq,
                                                nullptr, sw, make_ctx(stream, status, false),
                                                /*f64_rotation=*/true, (1 << (bits - 1)) - 1));
}

CK_API ck_status ck_rotate_quantize_act(const void *x, int64_t M, int64_t K, int64_t ldx,
                                        ck_input_act act, int g, int8_t *xq, float *sx,
                                        ck_stream_t stream) {
    CK_TRACE("ck_rotate_quantize_act");
    if (!x || !xq || !sx) return CK_ERR_NULL;
    if (act != CK_ACT_NONE && act != CK_ACT_SWIGLU) return CK_ERR_INVALID;
    if (M < 1 || K < 1 || M > kMaxRows || K > kMaxK) return CK_ERR_SHAPE;
    const int64_t need = act == CK_ACT_SWIGLU ? 2 * K : K;
    if (ldx < need || ldx % 8 != 0) return CK_ERR_SHAPE;
    if (!valid_group(g) || K % g != 0) return CK_ERR_GROUP;
    if (!aligned16(x) || !aligned16(xq)) return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    return from_cuda(ck::launch_rotate_quantize(
        x, false, act == CK_ACT_SWIGLU ? ck::Act::kSwiglu : ck::Act::kNone, g, M, K, ldx, xq,
        nullptr, sx, quant_ctx(stream, status, false)));
}

CK_API ck_status ck_rotate_quantize_act_f16(const void *x, int64_t M, int64_t K, int64_t ldx,
                                            ck_input_act act, int g, void *xq16, float *sx,
                                            ck_stream_t stream) {
    CK_TRACE("ck_rotate_quantize_act_f16");
    if (!x || !xq16 || !sx) return CK_ERR_NULL;
    if (act != CK_ACT_NONE && act != CK_ACT_SWIGLU) return CK_ERR_INVALID;
    if (M < 1 || K < 1 || M > kMaxRows || K > kMaxK) return CK_ERR_SHAPE;
    const int64_t need = act == CK_ACT_SWIGLU ? 2 * K : K;
    if (ldx < need || ldx % 8 != 0) return CK_ERR_SHAPE;
    if (!valid_group(g) || K % g != 0) return CK_ERR_GROUP;
    if (!aligned16(x) || !aligned16(xq16)) return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    return from_cuda(ck::launch_rotate_quantize(
        x, false, act == CK_ACT_SWIGLU ? ck::Act::kSwiglu : ck::Act::kNone, g, M, K, ldx, nullptr,
        xq16, sx, quant_ctx(stream, status, false)));
}

CK_API ck_status ck_int8_gemm_dequant(const void *xq16, const float *sx, int64_t M, int64_t K,
                                      const void *W, const float *sw, int64_t N,
                                      const void *bias, const void *residual, void *y,
                                      ck_stream_t stream) {
    CK_TRACE("ck_int8_gemm_dequant");
    if (!xq16 || !sx || !W || !sw || !y) return CK_ERR_NULL;
    if (M < 1 || N < 1 || K < 1 || M > kMaxRows || N > kMaxRows || K > kMaxK) return CK_ERR_SHAPE;
    if (K % 64 != 0 || N % 8 != 0) return CK_ERR_SHAPE;
    if (!aligned16(xq16) || !aligned16(W) || !aligned16(sw) || !aligned16(y) ||
        (bias && !aligned16(bias)) || (residual && !aligned16(residual)))
        return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    return from_cuda(ck::launch_gemm_codes(xq16, W, M, N, K, sx, sw, bias, residual, y, ck::kOutBf16,
                                           make_ctx(stream, status, g_overlap.load())));
}

CK_API size_t ck_prepared_weight_bytes(ck_wlayout layout, int64_t N, int64_t K) {
    if (N < 1 || K < 1) return 0;
    switch (layout) {
        case CK_WLAYOUT_ROWMAJOR_I8: return static_cast<size_t>(N) * K;
        case CK_WLAYOUT_GEMM_F16: return static_cast<size_t>(N) * K * 2;
        case CK_WLAYOUT_GEMM_F16_GLU: return N % 2 == 0 ? static_cast<size_t>(N) * K * 2 : 0;
        case CK_WLAYOUT_GEMV_PACKED: return K % 32 == 0 ? ck::gemv_packed_bytes(N, K) : 0;
        case CK_WLAYOUT_GEMV_PACKED_W6: return K % 32 == 0 ? ck::gemv_packed_lowbit_bytes(N, K, 6) : 0;
        case CK_WLAYOUT_GEMV_PACKED_W4: return K % 32 == 0 ? ck::gemv_packed_lowbit_bytes(N, K, 4) : 0;
    }
    return 0;
}

CK_API ck_status ck_prepare_weight(const int8_t *Wq, const float *sw, int64_t N, int64_t K,
                                   ck_wlayout layout, void *out, size_t out_bytes,
                                   ck_stream_t stream) {
    CK_TRACE("ck_prepare_weight");
    if (!Wq || !out) return CK_ERR_NULL;
    const int wbits = gemv_layout_bits(layout);
    if (layout != CK_WLAYOUT_ROWMAJOR_I8 && layout != CK_WLAYOUT_GEMM_F16 &&
        layout != CK_WLAYOUT_GEMM_F16_GLU && wbits == 0)
        return CK_ERR_INVALID;
    if (wbits != 0 && !sw) return CK_ERR_NULL;
    if (N < 1 || K < 1 || N > kMaxRows || K > kMaxK || K % 32 != 0) return CK_ERR_SHAPE;
    if (layout == CK_WLAYOUT_GEMM_F16_GLU && N % 2 != 0) return CK_ERR_SHAPE;
    if (!aligned16(Wq) || !aligned16(out)) return CK_ERR_ALIGN;
    if (out_bytes < ck_prepared_weight_bytes(layout, N, K)) return CK_ERR_WORKSPACE;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (layout) {
        case CK_WLAYOUT_ROWMAJOR_I8:
            return from_cuda(cudaMemcpyAsync(out, Wq, static_cast<size_t>(N) * K,
                                             cudaMemcpyDeviceToDevice, s));
        case CK_WLAYOUT_GEMM_F16: return from_cuda(ck::launch_widen_codes(Wq, N * K, out, s));
        case CK_WLAYOUT_GEMM_F16_GLU: return from_cuda(ck::launch_widen_codes_glu(Wq, N, K, out, s));
        case CK_WLAYOUT_GEMV_PACKED: return from_cuda(ck::launch_pack_gemv(Wq, sw, N, K, out, s));
        case CK_WLAYOUT_GEMV_PACKED_W6:
        case CK_WLAYOUT_GEMV_PACKED_W4:
            return from_cuda(ck::launch_pack_gemv_lowbit(Wq, sw, N, K, wbits, out, s));
    }
    return CK_ERR_INVALID;
}

CK_API size_t ck_workspace_bytes(ck_op op, int64_t M, int64_t K, int64_t N, ck_wlayout wlayout) {
    if (M < 1 || K < 1 || N < 1) return 0;
    switch (op) {
        case CK_OP_INT8_LINEAR: return linear_ws(M, K, N, wlayout).total;
        case CK_OP_SWIGLU_MLP: return mlp_ws(M, K, N, wlayout).total;
        case CK_OP_GEMV_SMALLM:
            return round_up(static_cast<size_t>(M) * K, 256) + round_up(static_cast<size_t>(M) * 4, 256);
        case CK_OP_DEBUG_GEMM_S32: return debug_ws(M, K, N).total;
    }
    return 0;
}

// One linear on prepared pieces: quantize x into codes16/scales, then the GEMM
// (launched as a programmatic dependent of the quantizer).  resident_weights:
// W16 is the caller's GEMM-resident weight, not a copy widened by this call.
static ck_status run_linear(const void *x, int64_t M, int64_t K, int64_t ldx, ck_input_act act,
                            const void *W16, const float *sw, int64_t N, int g, const void *bias,
                            const void *residual, void *y, void *xq16, float *sx,
                            unsigned int *status, ck_stream_t stream, bool resident_weights) {
    cudaError_t e = ck::launch_rotate_quantize(
        x, false, act == CK_ACT_SWIGLU ? ck::Act::kSwiglu : ck::Act::kNone, g, M, K, ldx, nullptr,
        xq16, sx, quant_ctx(stream, status, resident_weights));
    if (e != cudaSuccess) return CK_ERR_CUDA;
    e = ck::launch_gemm_codes(xq16, W16, M, N, K, sx, sw, bias, residual, y, ck::kOutBf16,
                              make_ctx(stream, status, true));
    return from_cuda(e);
}

CK_API ck_status ck_int8_linear(const void *x, int64_t M, int64_t K, int64_t ldx,
                                ck_input_act act, const void *W, ck_wlayout wlayout,
                                const float *sw, int64_t N, int g, const void *bias,
                                const void *residual, void *y, void *ws, size_t ws_bytes,
                                ck_stream_t stream) {
    CK_TRACE("ck_int8_linear");
    if (!x || !W || !sw || !y) return CK_ERR_NULL;
    if (wlayout != CK_WLAYOUT_ROWMAJOR_I8 && wlayout != CK_WLAYOUT_GEMM_F16) return CK_ERR_INVALID;
    if (ck_status st = check_linear_shape(M, K, ldx, act, N, g); st != CK_OK) return st;
    if (!aligned16(x) || !aligned16(W) || !aligned16(sw) || !aligned16(y) ||
        (bias && !aligned16(bias)) || (residual && !aligned16(residual)))
        return CK_ERR_ALIGN;
    const LinearWs plan = linear_ws(M, K, N, wlayout);
    if (!ws || ws_bytes < plan.total) return CK_ERR_WORKSPACE;
    if (!aligned16(ws)) return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    const void *W16 = W;
    if (wlayout == CK_WLAYOUT_ROWMAJOR_I8) {
        void *w16 = at<void>(ws, plan.w16);
        if (ck::launch_widen_codes(static_cast<const int8_t *>(W), N * K, w16,
                                   reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
            return CK_ERR_CUDA;
        W16 = w16;
    }
    return run_linear(x, M, K, ldx, act, W16, sw, N, g, bias, residual, y, at<void>(ws, plan.xq),
                      at<float>(ws, plan.sx), status, stream, wlayout == CK_WLAYOUT_GEMM_F16);
}

CK_API ck_status ck_swiglu_mlp(const void *x, int64_t M, int64_t H, int64_t I, const void *Wgu,
                               const float *sgu, const void *bgu, const void *Wd,
                               const float *sd, const void *bd, const void *residual,
                               ck_wlayout wlayout, int g, void *y, void *ws, size_t ws_bytes,
                               ck_stream_t stream) {
    CK_TRACE("ck_swiglu_mlp");
    if (!x || !Wgu || !sgu || !Wd || !sd || !y) return CK_ERR_NULL;
    if (wlayout != CK_WLAYOUT_ROWMAJOR_I8 && wlayout != CK_WLAYOUT_GEMM_F16 &&
        wlayout != CK_WLAYOUT_GEMM_F16_GLU)
        return CK_ERR_INVALID;
    if (ck_status st = check_linear_shape(M, H, H, CK_ACT_NONE, 2 * I, g); st != CK_OK) return st;
    if (ck_status st = check_linear_shape(M, I, 2 * I, CK_ACT_SWIGLU, H, g); st != CK_OK) return st;
    if (!aligned16(x) || !aligned16(Wgu) || !aligned16(sgu) || !aligned16(Wd) || !aligned16(sd) ||
        !aligned16(y) || (bgu && !aligned16(bgu)) || (bd && !aligned16(bd)) ||
        (residual && !aligned16(residual)))
        return CK_ERR_ALIGN;
    const MlpWs plan = mlp_ws(M, H, I, wlayout);
    if (!ws || ws_bytes < plan.total) return CK_ERR_WORKSPACE;
    if (!aligned16(ws)) return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *h = at<void>(ws, plan.h);
    const bool resident = wlayout != CK_WLAYOUT_ROWMAJOR_I8;
    if (wlayout == CK_WLAYOUT_GEMM_F16_GLU) {
        // SwiGLU in the gate|up GEMM's epilogue: it writes a = silu(gate) * up
        // in f32 (into the bytes h takes otherwise), which the down linear's
        // quantizer rotates and rounds as it would its own product
        void *xq16 = at<void>(ws, plan.xq);
        float *sx = at<float>(ws, plan.sx);
        if (ck::launch_rotate_quantize(x, false, ck::Act::kNone, g, M, H, H, nullptr, xq16, sx,
                                       quant_ctx(stream, status, true)) != cudaSuccess)
            return CK_ERR_CUDA;
        if (ck::launch_gemm_codes(xq16, Wgu, M, 2 * I, H, sx, sgu, bgu, nullptr, h, ck::kOutGlu,
                                  make_ctx(stream, status, true)) != cudaSuccess)
            return CK_ERR_CUDA;
        void *aq16 = at<void>(ws, plan.aq);
        float *sa = at<float>(ws, plan.sa);
        if (ck::launch_rotate_quantize(h, true, ck::Act::kGluF32, g, M, I, I, nullptr, aq16, sa,
                                       quant_ctx(stream, status, true)) != cudaSuccess)
            return CK_ERR_CUDA;
        return from_cuda(ck::launch_gemm_codes(aq16, Wd, M, H, I, sa, sd, bd, residual, y,
                                               ck::kOutBf16, make_ctx(stream, status, true)));
    }
    const void *Wgu16 = Wgu, *Wd16 = Wd;
    void *w16 = at<void>(ws, plan.w16);
    if (wlayout == CK_WLAYOUT_ROWMAJOR_I8) {
        if (ck::launch_widen_codes(static_cast<const int8_t *>(Wgu), 2 * I * H, w16, s) != cudaSuccess)
            return CK_ERR_CUDA;
        Wgu16 = w16;
    }
    ck_status st = run_linear(x, M, H, H, CK_ACT_NONE, Wgu16, sgu, 2 * I, g, bgu, nullptr, h,
                              at<void>(ws, plan.xq), at<float>(ws, plan.sx), status, stream,
                              resident);
    if (st != CK_OK) return st;
    if (wlayout == CK_WLAYOUT_ROWMAJOR_I8) {
        // stream order: the gate|up GEMM has consumed w16 before this overwrites it
        if (ck::launch_widen_codes(static_cast<const int8_t *>(Wd), H * I, w16, s) != cudaSuccess)
            return CK_ERR_CUDA;
        Wd16 = w16;
    }
    return run_linear(h, M, I, 2 * I, CK_ACT_SWIGLU, Wd16, sd, H, g, bd, residual, y,
                      at<void>(ws, plan.aq), at<float>(ws, plan.sa), status, stream, resident);
}

// The small-M GEMV over a packed layout of wbits-bit weight codes.
static ck_status gemv_smallM(const void *x, int64_t M, int64_t K, int64_t ldx, ck_input_act act,
                             const void *Wpacked, int wbits, int64_t N, int g, const void *bias,
                             const void *residual, void *y, void *ws, size_t ws_bytes,
                             ck_stream_t stream) {
    if (!x || !Wpacked || !y) return CK_ERR_NULL;
    if (ck_status st = check_linear_shape(M, K, ldx, act, N, g); st != CK_OK) return st;
    if (M > 8 || K % 32 != 0) return CK_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(Wpacked) || !aligned16(y) || (bias && !aligned16(bias)) ||
        (residual && !aligned16(residual)))
        return CK_ERR_ALIGN;
    const size_t need = ck_workspace_bytes(CK_OP_GEMV_SMALLM, M, K, N, CK_WLAYOUT_GEMV_PACKED);
    if (!ws || ws_bytes < need) return CK_ERR_WORKSPACE;
    if (!aligned16(ws)) return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    const int qmode = g_gemv_quant_mode.load();
    if (qmode != 1 && ck::gemv_fusable(M, K) && (qmode == 2 || gemv_fuse_by_default(M, K))) {
        // few enough activation elements for every CTA to quantize them itself:
        // one kernel, headed like the quantizer (a programmatic dependent of the
        // kernel ahead, reading x only after its wait)
        return from_cuda(ck::launch_gemv_fused(
            x, ldx, act == CK_ACT_SWIGLU ? ck::Act::kSwiglu : ck::Act::kNone, g, M, K, Wpacked, wbits,
            N, bias, residual, y, quant_ctx(stream, status, true)));
    }
    int8_t *xq = static_cast<int8_t *>(ws);
    float *sx = at<float>(ws, round_up(static_cast<size_t>(M) * K, 256));
    cudaError_t e = ck::launch_rotate_quantize(
        x, false, act == CK_ACT_SWIGLU ? ck::Act::kSwiglu : ck::Act::kNone, g, M, K, ldx, xq,
        nullptr, sx, quant_ctx(stream, status, true));
    if (e != cudaSuccess) return CK_ERR_CUDA;
    return from_cuda(ck::launch_gemv_packed(xq, sx, M, K, Wpacked, wbits, N, bias, residual, y,
                                            make_ctx(stream, status, true)));
}

static ck_status gemv_dequant(const int8_t *xq, const float *sx, int64_t M, int64_t K,
                              const void *Wpacked, int wbits, int64_t N, const void *bias,
                              const void *residual, void *y, ck_stream_t stream) {
    if (!xq || !sx || !Wpacked || !y) return CK_ERR_NULL;
    if (M < 1 || M > 8 || K < 32 || N < 1 || N > kMaxRows || K > kMaxK) return CK_ERR_SHAPE;
    if (K % 32 != 0 || N % 8 != 0) return CK_ERR_SHAPE;
    if (!aligned16(xq) || !aligned16(Wpacked) || !aligned16(y) || (bias && !aligned16(bias)) ||
        (residual && !aligned16(residual)))
        return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    return from_cuda(ck::launch_gemv_packed(xq, sx, M, K, Wpacked, wbits, N, bias, residual, y,
                                            make_ctx(stream, status, g_overlap.load())));
}

CK_API ck_status ck_int8_gemv_smallM(const void *x, int64_t M, int64_t K, int64_t ldx,
                                     ck_input_act act, const void *Wpacked, int64_t N, int g,
                                     const void *bias, const void *residual, void *y, void *ws,
                                     size_t ws_bytes, ck_stream_t stream) {
    CK_TRACE("ck_int8_gemv_smallM");
    return gemv_smallM(x, M, K, ldx, act, Wpacked, 8, N, g, bias, residual, y, ws, ws_bytes, stream);
}

CK_API ck_status ck_int8_gemv_dequant(const int8_t *xq, const float *sx, int64_t M, int64_t K,
                                      const void *Wpacked, int64_t N, const void *bias,
                                      const void *residual, void *y, ck_stream_t stream) {
    CK_TRACE("ck_int8_gemv_dequant");
    return gemv_dequant(xq, sx, M, K, Wpacked, 8, N, bias, residual, y, stream);
}

CK_API ck_status ck_packed_gemv_smallM(const void *x, int64_t M, int64_t K, int64_t ldx,
                                       ck_input_act act, const void *Wpacked, ck_wlayout wlayout,
                                       int64_t N, int g, const void *bias, const void *residual,
                                       void *y, void *ws, size_t ws_bytes, ck_stream_t stream) {
    CK_TRACE("ck_packed_gemv_smallM");
    const int wbits = gemv_layout_bits(wlayout);
    if (wbits == 0) return CK_ERR_INVALID;
    return gemv_smallM(x, M, K, ldx, act, Wpacked, wbits, N, g, bias, residual, y, ws, ws_bytes,
                       stream);
}

CK_API ck_status ck_packed_gemv_dequant(const int8_t *xq, const float *sx, int64_t M, int64_t K,
                                        const void *Wpacked, ck_wlayout wlayout, int64_t N,
                                        const void *bias, const void *residual, void *y,
                                        ck_stream_t stream) {
    CK_TRACE("ck_packed_gemv_dequant");
    const int wbits = gemv_layout_bits(wlayout);
    if (wbits == 0) return CK_ERR_INVALID;
    return gemv_dequant(xq, sx, M, K, Wpacked, wbits, N, bias, residual, y, stream);
}

CK_API ck_status ck_poll_device_status(ck_stream_t stream) {
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return CK_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return CK_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return CK_ERR_CUDA;
        return CK_ERR_TIMEOUT;
    }
    return CK_OK;
}

CK_API ck_status ck_debug_int8_gemm_s32(const int8_t *xq, const int8_t *Wq, int64_t M, int64_t N,
                                        int64_t K, int32_t *acc, void *ws, size_t ws_bytes,
                                        ck_stream_t stream) {
    if (!xq || !Wq || !acc) return CK_ERR_NULL;
    if (M < 1 || N < 1 || K < 1 || M > kMaxRows || N > kMaxRows || K > kMaxK) return CK_ERR_SHAPE;
    if (K % 64 != 0 || N % 8 != 0) return CK_ERR_SHAPE;
    if (!aligned16(xq) || !aligned16(Wq) || !aligned16(acc)) return CK_ERR_ALIGN;
    const DebugWs plan = debug_ws(M, K, N);
    if (!ws || ws_bytes < plan.total) return CK_ERR_WORKSPACE;
    if (!aligned16(ws)) return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *a16 = at<void>(ws, plan.a16);
    void *b16 = at<void>(ws, plan.b16);
    if (ck::launch_widen_codes(xq, M * K, a16, s) != cudaSuccess) return CK_ERR_CUDA;
    if (ck::launch_widen_codes(Wq, N * K, b16, s) != cudaSuccess) return CK_ERR_CUDA;
    return from_cuda(ck::launch_gemm_codes(a16, b16, M, N, K, nullptr, nullptr, nullptr, nullptr,
                                           acc, ck::kOutS32,
                                           make_ctx(stream, status, false)));
}

CK_API ck_status ck_debug_gemv_s32(const int8_t *xq, int64_t M, int64_t K, const void *Wpacked,
                                   ck_wlayout wlayout, int64_t N, int32_t *acc,
                                   ck_stream_t stream) {
    if (!xq || !Wpacked || !acc) return CK_ERR_NULL;
    const int wbits = gemv_layout_bits(wlayout);
    if (wbits == 0) return CK_ERR_INVALID;
    if (M < 1 || M > 8 || K < 32 || N < 1 || N > kMaxRows || K > kMaxK) return CK_ERR_SHAPE;
    if (K % 32 != 0 || N % 8 != 0) return CK_ERR_SHAPE;
    if (!aligned16(xq) || !aligned16(Wpacked) || !aligned16(acc)) return CK_ERR_ALIGN;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    return from_cuda(ck::launch_gemv_packed(xq, nullptr, M, K, Wpacked, wbits, N, nullptr, nullptr,
                                            nullptr, make_ctx(stream, status, false), acc));
}

CK_API void ck_debug_force_gemm_tile(int bn) { ck::set_forced_gemm_bn(bn); }

CK_API void ck_debug_force_gemv_quantizer(int mode) {
    g_gemv_quant_mode.store(mode == 1 || mode == 2 ? mode : 0);
}

CK_API ck_status ck_measure_int8_mma_tops(double *tops, int *sink, ck_stream_t stream) {
    if (!tops || !sink) return CK_ERR_NULL;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    return from_cuda(
        ck::measure_int8_mma_tops(tops, sink, reinterpret_cast<cudaStream_t>(stream)));
}

CK_API ck_status ck_measure_tcgen05_f16_tflops(double *tflops, ck_stream_t stream) {
    if (!tflops) return CK_ERR_NULL;
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    return from_cuda(ck::measure_tcgen05_f16_tflops(tflops, make_ctx(stream, status, false)));
}

CK_API int ck_debug_gemm_tile_choice(int64_t M, int64_t N, int64_t K, int sms) {
    if (M < 1 || N < 1 || K < 1 || sms < 2) return 0;
    return ck::gemm_tile_choice(M, N, K, sms);
}

CK_API ck_status ck_debug_stalled_wait(ck_stream_t stream) {
    unsigned int *status = nullptr;
    if (ck_status st = device_ready(&status); st != CK_OK) return st;
    return from_cuda(ck::launch_stalled_wait(make_ctx(stream, status, false)));
}

}  // extern "C"
