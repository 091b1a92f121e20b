// relayout.cu -- one-off weight relayouts into the resident layouts
// (comfy-kitchen PR #248, "Description": weight relayout facilities and the
// resident decode-layout hook).
//
// widen_codes: int8 codes -> the same integers as fp16 values, the operand
// format of the tcgen05 kind::f16 GEMM.  Exact: |q| <= 127 < 2^11.
// widen_codes_glu: the same for a packed [gate | up] weight, with its gate and
// up rows interleaved (the GEMM then forms silu(gate) * up in its epilogue).
#include <cuda_fp16.h>

#include "internal.h"

namespace ck {
namespace {

// 16 codes (one 16-byte load) -> 16 fp16 values (two 16-byte stores).
__device__ __forceinline__ void widen16(const int4 v, uint4 *dst) {
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
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

__global__ void widen_codes_kernel(const int8_t *__restrict__ q, int64_t n16,
                                   __half *__restrict__ out) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        widen16(__ldg(reinterpret_cast<const int4 *>(q) + i), reinterpret_cast<uint4 *>(out) + 2 * i);
}

// Output row r of the interleaved [gate | up] weight reads row r / 2
// (r even) or I + r / 2 (r odd); p16 = K / 16 pieces per row.
__global__ void widen_codes_glu_kernel(const int8_t *__restrict__ q, int64_t n16, int64_t p16,
                                       int64_t I, __half *__restrict__ out) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / p16, p = i % p16;
        const int64_t src = (r >> 1) + ((r & 1) ? I : 0);
        widen16(__ldg(reinterpret_cast<const int4 *>(q) + src * p16 + p),
                reinterpret_cast<uint4 *>(out) + 2 * i);
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

cudaError_t launch_widen_codes_glu(const int8_t *q, int64_t N, int64_t K, void *out16,
                                   cudaStream_t stream) {
    if (N <= 0 || K <= 0) return cudaSuccess;
    if (N % 2 != 0 || K % 16 != 0) return cudaErrorInvalidValue;
    const int64_t n16 = N * K / 16;
    int64_t blocks = (n16 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    widen_codes_glu_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        q, n16, K / 16, N / 2, static_cast<__half *>(out16));
    return cudaGetLastError();
}

}  // namespace ck
