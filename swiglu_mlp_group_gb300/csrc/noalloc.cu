// noalloc.cu -- ck_int8_linear_noalloc: the ConvRot linear for callers that
// cannot allocate device memory.  Its temporaries live in one file-scope
// device array instead of a caller workspace; no allocation happens anywhere
// on this path.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "ck.h"
#include "internal.h"
#include "trace.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kScratchBytes = CK_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device; held by each GPU that loads the library.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_dev[kMaxDevices] = {};  // device address of the array, per device

size_t round_up256(size_t v) { return (v + 255) / 256 * 256; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current.
ck_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return CK_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_dev[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return CK_ERR_CUDA;
        }
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return CK_OK;
}

}  // namespace

extern "C" CK_API ck_status ck_int8_linear_noalloc(const void *x, int64_t M, int64_t K,
                                                   int64_t ldx, ck_input_act act, const void *W16,
                                                   const float *sw, int64_t N, int g,
                                                   const void *bias, const void *residual,
                                                   void *y, ck_stream_t stream) {
    CK_TRACE("ck_int8_linear_noalloc");
    if (!x || !W16 || !sw || !y) return CK_ERR_NULL;
    if (act != CK_ACT_NONE && act != CK_ACT_SWIGLU) return CK_ERR_INVALID;
    if (M < 1 || K < 1 || N < 1 || M > INT32_MAX || N > INT32_MAX || K > 32768) return CK_ERR_SHAPE;
    const int64_t need_cols = act == CK_ACT_SWIGLU ? 2 * K : K;
    if (ldx < need_cols || ldx % 8 != 0 || N % 8 != 0) return CK_ERR_SHAPE;
    if ((g != 64 && g != 128 && g != 256) || K % g != 0) return CK_ERR_GROUP;
    if (!aligned16(x) || !aligned16(W16) || !aligned16(sw) || !aligned16(y) ||
        (bias && !aligned16(bias)) || (residual && !aligned16(residual)))
        return CK_ERR_ALIGN;
    const size_t codes_bytes = round_up256(static_cast<size_t>(M) * static_cast<size_t>(K) * 2);
    if (codes_bytes + static_cast<size_t>(M) * 4 > kScratchBytes) return CK_ERR_WORKSPACE;
    unsigned int *status = nullptr;
    if (const int st = ck::device_ready_status(&status); st != CK_OK)
        return static_cast<ck_status>(st);
    void *scratch = nullptr;
    if (const ck_status st = scratch_address(&scratch); st != CK_OK) return st;

    void *xq16 = scratch;
    float *sx = reinterpret_cast<float *>(static_cast<unsigned char *>(scratch) + codes_bytes);
    ck::LaunchCtx ctx;
    ctx.stream = reinterpret_cast<cudaStream_t>(stream);
    ctx.status = status;
    ctx.timeout_ns = ck::wait_timeout_ns();
    // the quantizer waits for the kernel ahead of it before touching memory;
    // W16 is the caller's GEMM-resident weight
    ctx.pdl = true;
    ctx.early_trigger = ck::launch_overlap();
    // the quantizer overwrites every code and scale the GEMM then reads
    if (ck::launch_rotate_quantize(x, false,
                                   act == CK_ACT_SWIGLU ? ck::Act::kSwiglu : ck::Act::kNone, g, M,
                                   K, ldx, nullptr, xq16, sx, ctx) != cudaSuccess)
        return CK_ERR_CUDA;
    ctx.early_trigger = false;
    return ck::launch_gemm_codes(xq16, W16, M, N, K, sx, sw, bias, residual, y, ck::kOutBf16, ctx) ==
                   cudaSuccess
               ? CK_OK
               : CK_ERR_CUDA;
}
