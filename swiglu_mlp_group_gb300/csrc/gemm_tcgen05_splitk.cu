// gemm_tcgen05_splitk.cu -- the CTA-pair GEMM of gemm_tcgen05_2sm.cu with K
// split between the two pairs of a four-CTA cluster, for problems with too
// few 256 x 256 tiles to fill the GPU's pairs (the linear step's
// 2048 x 3072 -> 1024 has 32 of them on 76 pairs):
//
//   acc[m, n] = sum_{k < K0} xq[m, k] Wq[n, k] + sum_{k >= K0} xq[m, k] Wq[n, k]
//   y[m, n]   = bf16( f32(acc) * sx[m] * sw[n] + bias[n] + residual[m, n] )
// (comfy-kitchen PR #277, "Summary" / "The key observation"); both halves are
// exact int32 sums, so their sum is the GEMM's exact result.
//
// Why: each SM of a pair takes in its operand stages at a bounded rate, so the
// k-loop of a tile costs about K / 64 times a stage's bytes over that rate.
// With one round of 256 x 128 pair tiles on 128 SMs the small shape spends
// 10 us there; 256 x 256 tiles halve the operand bytes per product, and the
// split halves each SM's share of K.
//
// Cluster ranks: 0, 1 = pair 0 (k-blocks [0, nkb / 2)), 2, 3 = pair 1 (the
// rest); the even CTA of each pair issues its MMAs.  One cluster per tile
// (not persistent).  Within a pair everything is the pair kernel's: the
// producer, the single-lane MMA issuer, the 1024-product f32 chunks drained to
// int32 registers by eight epilogue warps (thread (warp w, lane l): row
// 32 (w % 4) + l of the CTA's 128, columns 128 h .. 128 h + 127 of the tile,
// h = (w - 2) / 4).
//
// Combining the halves, column-wise: pair p finishes columns 128 p .. 128 p +
// 127 of the tile, on all eight epilogue warps (64 columns each, the stores
// coalesced as in the 64-column-half kernels).  After its last chunk:
//  - the warps holding the partner's columns stage their int32 sums in their
//    own stage ring (free now), and one bulk copy (TMA, shared to shared
//    memory of the cluster) moves the 64 KB into the partner's ring, counted
//    in bytes on its exchange barrier, once the partner has reported its ring
//    free (a cluster-scope arrive);
//  - each warp holding this pair's columns hands the upper 64 of them to its
//    twin (the warp of the same rows) through shared memory;
//  - every warp adds the partner's sums of its 64 columns and dequantizes.
// Every wait is bounded (gemm_tcgen05.cu).
#include <cuda_bf16.h>

#include "gemm_epilogue.cuh"
#include "gemm_issue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"

namespace ck {
namespace {

constexpr int kRows = 128;                 // A rows per CTA (pair tile: 256 rows)
constexpr int kBK = 64;
constexpr int kPN = 256;                   // pair tile width
constexpr int kCols = kPN / 2;             // columns per epilogue thread
constexpr int kABytes = kRows * kBK * 2;   // 16 KB
constexpr int kBBytes = (kPN / 2) * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStages = 6;
constexpr int kTmemCols = 512;             // two 256-column accumulator buffers
constexpr int kThreads = 320;
constexpr int kChunkBlocks = 16;           // 1024 products per f32 chunk
constexpr int kBarBytes = 256;
constexpr int kFin = kCols / 2;           // columns each epilogue thread finishes
constexpr uint32_t kXBytes = 4 * 32 * kCols * 4;  // int32 sums one CTA receives: 64 KB
constexpr int kXInOff = 0;                 // ring regions of the exchange (see the epilogue)
constexpr int kHandOff = kXBytes;
constexpr int kXOutOff = kXBytes + kXBytes / 2;
constexpr int kSendBarId = 2;              // named barriers (1 is the epilogue's)
constexpr int kTwinBarId0 = 3;             // 3 .. 6: the two warps of row block q
constexpr size_t kSmemBytes =
    static_cast<size_t>(kStages) * kStageBytes + kBarBytes + ep::staging_bytes(kPN) + 1024;
static_assert(kXOutOff + kXBytes <= static_cast<uint32_t>(kStages) * kStageBytes, "exchange must fit the ring");

// try_wait whose completion acquires at cluster scope: the phases completed by
// another CTA (a release.cluster arrive, a bulk copy's bytes).
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// mbar_wait (time bound, abort flag) on such a phase.
__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
    if (try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (try_wait_cluster(bar, parity)) return true;
        if (*ctl.abort_flag) return false;
        if (globaltimer_ns() - t0 > ctl.timeout_ns) {
            *ctl.abort_flag = 1;
            atomicOr(ctl.status, kDeviceStatusTimeout);
            return false;
        }
    }
}
// Generic-proxy writes to this CTA's shared memory become visible to the
// async proxy (a bulk copy reading them).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// this CTA's shared memory to another CTA's (cluster address), counted in
// bytes on that CTA's barrier bar_cluster.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                     uint32_t bar_cluster) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst_cluster),
                 "r"(src), "r"(bytes), "r"(bar_cluster)
                 : "memory");
}

template <int OUT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_codes_splitk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         int M, int N, int K, int m_pairs, const float *__restrict__ sx,
                         const float *__restrict__ sw, const __nv_bfloat16 *__restrict__ bias,
                         const __nv_bfloat16 *residual, void *out, unsigned int *status,
                         unsigned long long timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t smem_s = raw_s + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    const uint32_t bars_s = smem_s + kStages * kStageBytes;
    auto full_bar = [&](int s) { return bars_s + 8u * s; };
    auto empty_bar = [&](int s) { return bars_s + 8u * (kStages + s); };
    auto accf_bar = [&](int b) { return bars_s + 8u * (2 * kStages + b); };
    auto acce_bar = [&](int b) { return bars_s + 8u * (2 * kStages + 2 + b); };
    const uint32_t done_bar = bars_s + 8u * (2 * kStages + 4);
    const uint32_t xfree_bar = bars_s + 8u * (2 * kStages + 5);  // the partner's ring is free
    const uint32_t xdata_bar = bars_s + 8u * (2 * kStages + 6);  // the partner's sums are here
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kStages + 7);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *ep_sw = reinterpret_cast<float *>(smem + kStages * kStageBytes + kBarBytes);
    float *ep_b = ep_sw + kPN;
    auto sA = [&](int s) { return smem_s + s * kStageBytes; };
    auto sB = [&](int s) { return smem_s + s * kStageBytes + kABytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t ks = rank >> 1;         // which half of K this pair sums
    const uint32_t prank = rank & 1u;      // 0: the pair's MMA issuer
    const uint32_t lead = rank & ~1u;      // the pair's even CTA
    const uint32_t partner = rank ^ 2u;    // same rows, other half of K
    const int tile = static_cast<int>(blockIdx.x >> 2);
    const int m_base = (tile % m_pairs) * (2 * kRows) + static_cast<int>(prank) * kRows;
    const int n_base = (tile / m_pairs) * kPN;
    const int num_kb = K / kBK;
    const int kb0 = ks == 0 ? 0 : num_kb / 2;
    const int nkb = ks == 0 ? num_kb / 2 : num_kb - num_kb / 2;
    const int nchunks = (nkb + kChunkBlocks - 1) / kChunkBlocks;
    const WaitCtl ctl{abort_flag, status, timeout_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 16);  // 8 epilogue warps in each CTA of the pair
        }
        mbar_init(done_bar, 1);
        mbar_init(xfree_bar, 1);
        mbar_init(xdata_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        // the partner's bulk copy completes the phase with these bytes
        mbar_arrive_expect_tx(xdata_bar, kXBytes);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // every CTA's barriers exist before any other CTA uses them
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const int a_row = m_base;
        const int b_row = n_base + static_cast<int>(prank) * (kPN / 2);
        const int pre = min(kStages, nkb);
        if (elect_one()) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            for (int kb = 0; kb < pre; ++kb) {
                if (prank == 0) mbar_arrive_expect_tx(full_bar(kb), 2 * kStageBytes);
                tma_load_2d_pair(sB(kb), &tmB, mapa_shared(full_bar(kb), lead), (kb0 + kb) * kBK, b_row);
            }
        }
        __syncwarp();
        pdl_wait();  // A (the activation codes) comes from the previous kernel
        int issued = 0;
        produce_loop<kStages>(
            nkb, nkb, pre, tile, 1, empty_bar(0), ctl,
            [&](int, int &ar, int &br) {
                ar = a_row;
                br = b_row;
            },
            [&](int st, int kb, int ar, int br, bool whole) {
                const uint32_t lead_full = mapa_shared(full_bar(st), lead);
                if (whole) {
                    if (prank == 0) mbar_arrive_expect_tx(full_bar(st), 2 * kStageBytes);
                    tma_load_2d_pair(sB(st), &tmB, lead_full, (kb0 + kb) * kBK, br);
                }
                tma_load_2d_pair(sA(st), &tmA, lead_full, (kb0 + kb) * kBK, ar);
            },
            issued);
        if (*abort_flag && elect_one()) {
            if (prank == 0) {
                const int first = issued > kStages ? issued - kStages : 0;
                for (int i = first; i < issued; ++i)
                    mbar_wait_drain(full_bar(i % kStages), (i / kStages) & 1, timeout_ns, status);
            } else {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 50000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (prank == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(2 * kRows, kPN);
            const uint16_t pair_mask = static_cast<uint16_t>(0x3u << lead);
            const uint16_t lead_mask = static_cast<uint16_t>(0x1u << lead);
            const IssueBars ib{full_bar(0), empty_bar(0), accf_bar(0), acce_bar(0)};
            issue_mma_loop<kStages, kChunkBlocks, kStageBytes / 16>(
                nkb, nkb, tmem_base, kPN, ib, sdesc_kmajor_sw128(sA(0)), sdesc_kmajor_sw128(sB(0)), ctl,
                [](uint32_t d, uint64_t a, uint64_t b, uint32_t acc) { mma_f16_ss_pair(d, a, b, idesc, acc); },
                [pair_mask](uint32_t bar) { mma_commit_pair(bar, pair_mask); });
            if (elect_one()) {
                mma_commit_pair(done_bar, lead_mask);
                mbar_wait_drain(done_bar, 0, timeout_ns, status);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const int et = threadIdx.x - 64;  // 0..255 over the epilogue warps
        const int slot = q * 32 + lane;   // this thread's place in the exchange
        const bool keeps = h == static_cast<int>(ks);  // holds columns finished in this pair
        float s_x = 0.f;
        if constexpr (OUT != kOutS32) {
            pdl_wait();  // sx comes from the previous kernel
            ep::stage(ep_sw, ep_b, et, kPN, n_base, N, sw, bias);
            const int m_row = m_base + slot;
            s_x = m_row < M ? sx[m_row] : 0.f;
        }
        bool ok = true;
        int32_t acc[kCols];
#pragma unroll
        for (int i = 0; i < kCols; ++i) acc[i] = 0;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int buf = c & 1;
            int got = 0;
            if (lane == 0) got = mbar_wait(accf_bar(buf), (c >> 1) & 1, ctl) ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(buf * kPN + h * kCols);
#pragma unroll
            for (int p = 0; p < kCols / 32; ++p) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + 32u * p, r);
                tmem_wait_ld(r);
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[p * 32 + i] += __float2int_rn(__uint_as_float(r[i]));
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(acce_bar(buf), lead));
        }
        // Once this pair's MMAs are over (this warp has the last chunk) the ring
        // holds, piece j (16 bytes) of thread `slot` at 16 (128 j + slot):
        //   xin  [0, 64 KB):    the partner's sums of the columns finished here
        //   hand [64, 96 KB):   the keeping warp's upper 64 columns, for its twin
        //   xout [96, 160 KB):  this CTA's sums of the partner's columns
        // Columns 128 ks .. 128 ks + 127 are finished here, the keeping warp
        // (q, ks) taking the first 64, its twin (q, 1 - ks) the other 64.
        const uint32_t pos = 16u * static_cast<uint32_t>(slot);
        int32_t fin[kFin];
        if (keeps) {
            if (ok && q == 0 && lane == 0) mbar_arrive_cluster(mapa_shared(xfree_bar, partner));
            if (ok) {
#pragma unroll
                for (int j = 0; j < kFin / 4; ++j)
                    *reinterpret_cast<int4 *>(smem + kHandOff + pos + 2048 * j) =
                        make_int4(acc[kFin + 4 * j], acc[kFin + 4 * j + 1], acc[kFin + 4 * j + 2],
                                  acc[kFin + 4 * j + 3]);
            }
#pragma unroll
            for (int i = 0; i < kFin; ++i) fin[i] = acc[i];
        } else {
            if (ok) {
#pragma unroll
                for (int j = 0; j < kCols / 4; ++j)
                    *reinterpret_cast<int4 *>(smem + kXOutOff + pos + 2048 * j) =
                        make_int4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
                fence_proxy_async_smem();  // visible to the bulk copy below
            }
            // all four sending warps have staged theirs; one of them sends the
            // 64 KB once the partner's ring is free
            const bool staged = !named_bar_or(kSendBarId, 128, !ok);
            ok = ok && staged;
            if (ok && q == 0) {
                ok = __all_sync(0xffffffffu, wait_cluster(xfree_bar, 0, ctl));
                if (ok && elect_one()) {
                    const uint32_t bar = mapa_shared(xdata_bar, partner);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        bulk_copy_to_cluster(mapa_shared(smem_s + kXInOff + c * (kXBytes / 4), partner),
                                             smem_s + kXOutOff + c * (kXBytes / 4), kXBytes / 4, bar);
                }
                __syncwarp();
            }
        }
        // the keeping warp's hand-off reaches its twin
        named_bar_sync(kTwinBarId0 + q, 64);
        if (!keeps && ok) {
#pragma unroll
            for (int j = 0; j < kFin / 4; ++j) {
                const int4 v = *reinterpret_cast<const int4 *>(smem + kHandOff + pos + 2048 * j);
                fin[4 * j] = v.x;
                fin[4 * j + 1] = v.y;
                fin[4 * j + 2] = v.z;
                fin[4 * j + 3] = v.w;
            }
        }
        // the partner's sums: every lane acquires the phase before reading them
        if (ok) ok = __all_sync(0xffffffffu, wait_cluster(xdata_bar, 0, ctl));
        const int half = keeps ? 0 : 1;
        if (ok) {
#pragma unroll
            for (int j = 0; j < kFin / 4; ++j) {
                const int4 v =
                    *reinterpret_cast<const int4 *>(smem + kXInOff + pos + 2048 * (half * (kFin / 4) + j));
                fin[4 * j] += v.x;
                fin[4 * j + 1] += v.y;
                fin[4 * j + 2] += v.z;
                fin[4 * j + 3] += v.w;
            }
        }
        // every epilogue thread passes this barrier, so a wait that gave up
        // anywhere stops all of them (and publishes the staged scales)
        ok = ep::sync_all_ok(ok);
        if (ok) {
            const int c0 = static_cast<int>(ks) * kCols + half * kFin;  // first column within the tile
            const int n0 = n_base + c0;
            if constexpr (OUT == kOutS32) {
                const int m = m_base + slot;
                if (m < M) {
                    int32_t *o = static_cast<int32_t *>(out) + static_cast<int64_t>(m) * N + n0;
#pragma unroll
                    for (int j = 0; j < kFin / 4; ++j)
                        if (n0 + 4 * j < N)
                            *reinterpret_cast<int4 *>(o + 4 * j) =
                                make_int4(fin[4 * j], fin[4 * j + 1], fin[4 * j + 2], fin[4 * j + 3]);
                }
            } else {
                ep::dequant_store<kFin>(fin, m_base + q * 32, lane, M, n0, N, s_x, ep_sw + c0, ep_b + c0,
                                        residual, static_cast<__nv_bfloat16 *>(out));
            }
        } else {
            // a copy the partner may still have in flight lands before this CTA exits
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 50000ull) {
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // MMAs, exchanges and remote arrives of the cluster are over
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

bool encode_f16(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows) {
    return tensor_map_2d(map, ptr, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rows, K, kBK, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int OUT>
cudaLaunchConfig_t splitk_config(int tiles, const LaunchCtx &ctx, cudaLaunchAttribute (&attr)[2]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(4 * tiles));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = ctx.stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ctx.pdl ? 2 : 1;
    return cfg;
}

template <int OUT>
cudaError_t launch_splitk_t(const void *A16, const void *B16, int64_t M, int64_t N, int64_t K, const float *sx,
                            const float *sw, const void *bias, const void *residual, void *out,
                            const LaunchCtx &ctx) {
    CUtensorMap ma, mb;
    if (!encode_f16(&ma, A16, M, K, kRows) || !encode_f16(&mb, B16, N, K, kPN / 2))
        return cudaErrorInvalidValue;
    auto kern = gemm_codes_splitk_kernel<OUT>;
    if (cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), static_cast<int>(kSmemBytes));
        e != cudaSuccess)
        return e;
    const int m_pairs = static_cast<int>((M + 2 * kRows - 1) / (2 * kRows));
    const int tiles = m_pairs * static_cast<int>((N + kPN - 1) / kPN);
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = splitk_config<OUT>(tiles, ctx, attr);
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, static_cast<int>(M), static_cast<int>(N),
                              static_cast<int>(K), m_pairs, sx, sw, static_cast<const __nv_bfloat16 *>(bias),
                              static_cast<const __nv_bfloat16 *>(residual), out, ctx.status,
                              static_cast<unsigned long long>(ctx.timeout_ns));
}

}  // namespace

int splitk_resident_clusters() {
    auto kern = gemm_codes_splitk_kernel<kOutBf16>;
    if (ensure_dynamic_smem(reinterpret_cast<const void *>(kern), static_cast<int>(kSmemBytes)) != cudaSuccess)
        return 0;
    return max_active_clusters(reinterpret_cast<const void *>(kern), kThreads, kSmemBytes, 4);
}

cudaError_t launch_gemm_codes_splitk(const void *A16, const void *B16, int64_t M, int64_t N, int64_t K,
                                     const float *sx, const float *sw, const void *bias, const void *residual,
                                     void *out, int out_kind, const LaunchCtx &ctx) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (K % kBK != 0 || K / kBK < 2) return cudaErrorInvalidValue;
    if (out_kind == kOutS32)
        return launch_splitk_t<kOutS32>(A16, B16, M, N, K, sx, sw, bias, residual, out, ctx);
    if (out_kind == kOutBf16)
        return launch_splitk_t<kOutBf16>(A16, B16, M, N, K, sx, sw, bias, residual, out, ctx);
    return cudaErrorInvalidValue;
}

}  // namespace ck
