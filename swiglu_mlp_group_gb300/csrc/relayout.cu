// relayout.cu -- one-off weight relayouts into the resident layouts
// (comfy-kitchen PR #248, "Description": weight relayout facilities and the
// resident decode-layout hook).
//
// widen_codes: int8 codes -> the same integers as fp16 values, the operand
// format of the tcgen05 kind::f16 GEMM.  Exact: |q| <= 127 < 2^11.
#include <cuda_fp16.h>

#include "internal.h"

namespace ck {
namespace {

// 16 codes per thread: one 16-byte load, two 16-byte stores.
__global__ void widen_codes_kernel(const int8_t *__restrict__ q, int64_t n16,
                                   __half *__restrict__ out) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int4 v = __ldg(reinterpret_cast<const int4 *>(q) + i);
        const int w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int lo = static_cast<int8_t>((w[j] >> (16 * b)) & 0xff);
                const int hi = static_cast<int8_t>((w[j] >> (16 * b + 8)) & 0xff);
                o[2 * j + b] = __half_as_ushort(__int2half_rn(lo)) |
                               (static_cast<uint32_t>(__half_as_ushort(__int2half_rn(hi))) << 16);
            }
        }
        uint4 *dst = reinterpret_cast<uint4 *>(out) + 2 * i;
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

}  // namespace

cudaError_t launch_widen_codes(const int8_t *q, int64_t n, void *out16, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int64_t n16 = n / 16;
    int64_t blocks = (n16 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    widen_codes_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        q, n16, static_cast<__half *>(out16));
    return cudaGetLastError();
}

}  // namespace ck
