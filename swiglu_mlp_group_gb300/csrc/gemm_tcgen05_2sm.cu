// gemm_tcgen05_2sm.cu -- the exact-integer ConvRot GEMM of gemm_tcgen05.cu on
// CTA pairs: tcgen05.mma.cta_group::2 computes a 256 x PN output tile
// (PN = 256, 224 or 128) on two SMs at once.
//
//   acc[m, n] = sum_k xq[m, k] * Wq[n, k]           (exact int32)
//   y[m, n]   = bf16( f32(acc) * sx[m] * sw[n] + bias[n] + residual[m, n] )
// (comfy-kitchen PR #277, "Summary" / "The key observation").
//
// Why pairs: each SM holds its 128 rows of A and half of B, so an SM moves
// less operand data through TMA and shared memory per unit of work than with
// one-SM tiles (measured on GB300: 4096^3 in 76 us on 224-column pair tiles
// against 97 us on one-SM 128 x 256 tiles; 4096 x 3072 -> 24576 326 against
// 357 us).
//
// Roles (each CTA of the pair, 10 warps):
//   warp 0     : TMA producer -- this CTA's A half (128 rows) and B half
//                (PN / 2 rows) of 64 K-columns; completion counted on the even
//                ("leader") CTA's full barrier (cp.async.bulk.tensor
//                .cta_group::2), stage reuse gated by this CTA's empty barrier.
//   warp 1     : TMEM allocation for the pair; in the leader only, the MMA
//                issuer (M = 256, N = PN, K = 16; one elected lane issues,
//                gemm_issue.cuh), whose commits release the stage and
//                publish the accumulator in both CTAs (multicast).
//   warps 2..9 : epilogue on this CTA's 128 rows, as in the one-CTA kernel;
//                buffer release is an arrive on the leader's barrier.
// Exactness, chunking (1024 K per f32 TMEM chunk, two alternating buffers),
// persistence over tiles and the bounded waits are those of gemm_tcgen05.cu.
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
constexpr int kABytes = kRows * kBK * 2;   // 16 KB
constexpr int kThreads = 320;
constexpr int kChunkBlocks = 16;           // 1024 products per f32 chunk

// Pair tile of 256 rows x PN columns (PN = 256, 224 or 128); each CTA holds PN / 2
// rows of B.  The width is picked per problem to balance the rounds of tiles.
template <int PN>
struct PairCfg {
    static constexpr int kBBytes = (PN / 2) * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = PN == 256 ? 6 : (PN == 224 ? 7 : 8);
    static constexpr int kTmemCols = PN > 128 ? 512 : 256;  // two PN-column accumulator buffers
    static constexpr int kBarBytes = 256;
    // stage ring, barriers, the epilogue's staged scales, alignment slack
    static constexpr size_t kSmemBytes =
        static_cast<size_t>(kStages) * kStageBytes + kBarBytes + ep::staging_bytes(PN) + 1024;
};

template <int PN, int OUT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_codes_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, int M, int N, int K, int m_pairs,
                       const float *__restrict__ sx, const float *__restrict__ sw,
                       const __nv_bfloat16 *__restrict__ bias, const __nv_bfloat16 *residual, void *out,
                       unsigned int *status, unsigned long long timeout_ns) {
    using Cfg = PairCfg<PN>;
    constexpr int kStages = Cfg::kStages;
    constexpr int kStageBytes = Cfg::kStageBytes;
    constexpr int kTmemCols = Cfg::kTmemCols;
    constexpr int kPairN = PN;
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
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kStages + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *ep_sw = reinterpret_cast<float *>(smem + kStages * kStageBytes + Cfg::kBarBytes);
    float *ep_b = ep_sw + kPairN;
    auto sA = [&](int s) { return smem_s + s * kStageBytes; };
    auto sB = [&](int s) { return smem_s + s * kStageBytes + kABytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: leader (issues the MMAs), 1: peer
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int total_tiles = m_pairs * ((N + kPairN - 1) / kPairN);
    const int num_kb = K / kBK;
    const int nchunks = (num_kb + kChunkBlocks - 1) / kChunkBlocks;
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
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before either uses the other's
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // A kernel queued behind this one may launch now: it waits for our end
    // before it touches anything we read or write.
    pdl_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const int my_tiles = pair < total_tiles ? (total_tiles - 1 - pair) / npairs + 1 : 0;
        const int total_kb = my_tiles * num_kb;
        const int half_rank = static_cast<int>(rank);
        // The weights do not depend on the previous kernel: the first stages'
        // B tiles are requested before waiting on it, A after.
        const int pre = total_kb > 0 ? min(kStages, num_kb) : 0;
        if (elect_one()) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            for (int kb = 0; kb < pre; ++kb) {
                if (rank == 0) mbar_arrive_expect_tx(full_bar(kb), 2 * kStageBytes);
                tma_load_2d_pair(sB(kb), &tmB, mapa_shared(full_bar(kb), 0), kb * kBK,
                                 (pair / m_pairs) * kPairN + half_rank * (kPairN / 2));
            }
        }
        __syncwarp();
        pdl_wait();  // A (the activation codes) comes from the previous kernel
        int issued = 0;
        // both CTAs' copies complete on the leader's full barrier, which counts
        // the pair's bytes; a stage is reused once the leader's MMAs released it
        produce_loop<kStages>(
            total_kb, num_kb, pre, pair, npairs, empty_bar(0), ctl,
            [&](int tile, int &a_row, int &b_row) {
                a_row = (tile % m_pairs) * (2 * kRows) + half_rank * kRows;
                b_row = (tile / m_pairs) * kPairN + half_rank * (kPairN / 2);
            },
            [&](int st, int kb, int a_row, int b_row, bool whole) {
                const uint32_t lead_full = mapa_shared(full_bar(st), 0);
                if (whole) {
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(st), 2 * kStageBytes);
                    tma_load_2d_pair(sB(st), &tmB, lead_full, kb * kBK, b_row);
                }
                tma_load_2d_pair(sA(st), &tmA, lead_full, kb * kBK, a_row);
            },
            issued);
        if (*abort_flag && elect_one()) {
            if (rank == 0) {
                // the leader's full barriers count both CTAs' bytes
                const int first = issued > kStages ? issued - kStages : 0;
                for (int i = first; i < issued; ++i)
                    mbar_wait_drain(full_bar(i % kStages), (i / kStages) & 1, timeout_ns, status);
            } else {
                // copies in flight into this CTA land within microseconds
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 50000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (rank == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(2 * kRows, kPairN);
            const int my_tiles = pair < total_tiles ? (total_tiles - 1 - pair) / npairs + 1 : 0;
            const IssueBars ib{full_bar(0), empty_bar(0), accf_bar(0), acce_bar(0)};
            // commits free the stage / publish the accumulator in both CTAs
            issue_mma_loop<kStages, kChunkBlocks, Cfg::kStageBytes / 16>(
                my_tiles * num_kb, num_kb, tmem_base, kPairN, ib, sdesc_kmajor_sw128(sA(0)),
                sdesc_kmajor_sw128(sB(0)), ctl,
                [](uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
                    mma_f16_ss_pair(d, a, b, idesc, acc);
                },
                [](uint32_t bar) { mma_commit_pair(bar, 0x3); });
            // no MMA may be in flight when TMEM is released (the commit comes
            // from the lane that issued them)
            if (elect_one()) {
                mma_commit_pair(done_bar, 0x1);
                mbar_wait_drain(done_bar, 0, timeout_ns, status);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        constexpr int kCols = kPairN / 2;
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const int et = threadIdx.x - 64;  // 0..255 over the epilogue warps
        float s_x = 0.f;  // this thread's row scale in the current tile
        if constexpr (OUT != kOutS32) pdl_wait();  // sx comes from the previous kernel
        bool ok = true;
        int gc = 0;
        for (int tile = pair; tile < total_tiles; tile += npairs) {
            const int m_base = (tile % m_pairs) * (2 * kRows) + static_cast<int>(rank) * kRows;
            const int n_base = (tile / m_pairs) * kPairN;
            if constexpr (OUT != kOutS32) {
                ep::sync();  // the previous tile's dequant no longer reads the staging
                if constexpr (OUT == kOutGlu)
                    ep::stage_glu(ep_sw, ep_b, et, kPairN, n_base, N, sw, bias);
                else
                    ep::stage(ep_sw, ep_b, et, kPairN, n_base, N, sw, bias);
                const int m_row = m_base + q * 32 + lane;
                s_x = m_row < M ? sx[m_row] : 0.f;
            }
            int32_t acc[kCols];
#pragma unroll
            for (int i = 0; i < kCols; ++i) acc[i] = 0;
            for (int c = 0; c < nchunks && ok; ++c, ++gc) {
                const int buf = gc & 1;
                int got = 0;
                if (lane == 0) got = mbar_wait(accf_bar(buf), (gc >> 1) & 1, ctl) ? 1 : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(buf * kPairN + h * kCols);
#pragma unroll
                for (int p = 0; p < kCols / 32; ++p) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + 32u * p, r);
                    tmem_wait_ld(r);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        acc[p * 32 + i] += __float2int_rn(__uint_as_float(r[i]));
                }
                if constexpr (kCols % 32 != 0) {  // PN = 224
                    static_assert(kCols % 32 == 16, "pair tile half-width must be 16 mod 32");
                    constexpr int p0 = kCols / 32 * 32;
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(tbase + p0, r);
                    tmem_wait_ld16(r);
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[p0 + i] += __float2int_rn(__uint_as_float(r[i]));
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(acce_bar(buf), 0));
            }
            const int n0 = n_base + h * kCols;
            if constexpr (OUT == kOutS32) {
                if (!ok) break;
                const int m = m_base + q * 32 + lane;
                if (m < M) {
                    int32_t *o = static_cast<int32_t *>(out) + static_cast<int64_t>(m) * N + n0;
#pragma unroll
                    for (int j = 0; j < kCols / 4; ++j) {
                        if (n0 + 4 * j < N)
                            *reinterpret_cast<int4 *>(o + 4 * j) =
                                make_int4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
                    }
                }
            } else {
                // every epilogue thread passes both barriers of a tile, so they
                // leave the loop together when any wait gave up
                ok = ep::sync_all_ok(ok);
                if (!ok) break;
                if constexpr (OUT == kOutGlu)
                    ep::glu_store<kCols>(acc, m_base + q * 32, lane, M, n0, N, s_x, ep_sw + h * kCols,
                                         ep_b + h * kCols, static_cast<float *>(out));
                else
                    ep::dequant_store<kCols>(acc, m_base + q * 32, lane, M, n0, N, s_x,
                                             ep_sw + h * kCols, ep_b + h * kCols, residual,
                                             static_cast<__nv_bfloat16 *>(out));
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // the leader's MMAs and both CTAs' barrier traffic are over
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

bool encode_f16(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows) {
    return tensor_map_2d(map, ptr, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rows, K, kBK, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int PN, int OUT>
cudaError_t launch_pair_t(const void *A16, const void *B16, int64_t M, int64_t N, int64_t K,
                          const float *sx, const float *sw, const void *bias, const void *residual, void *out,
                          const LaunchCtx &ctx) {
    using Cfg = PairCfg<PN>;
    CUtensorMap ma, mb;
    if (!encode_f16(&ma, A16, M, K, kRows) || !encode_f16(&mb, B16, N, K, PN / 2))
        return cudaErrorInvalidValue;
    auto kern = gemm_codes_pair_kernel<PN, OUT>;
    // the shared-memory opt-in belongs to each device's copy of the kernel
    if (cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                            static_cast<int>(Cfg::kSmemBytes));
        e != cudaSuccess)
        return e;
    const int sms = sm_count();
    if (sms < 2) return cudaErrorInvalidDevice;
    const int m_pairs = static_cast<int>((M + 2 * kRows - 1) / (2 * kRows));
    const int n_tiles = static_cast<int>((N + PN - 1) / PN);
    const int tiles = m_pairs * n_tiles;
    const int pairs = tiles < sms / 2 ? tiles : sms / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ctx.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, static_cast<int>(M), static_cast<int>(N),
                              static_cast<int>(K), m_pairs, sx, sw,
                              static_cast<const __nv_bfloat16 *>(bias),
                              static_cast<const __nv_bfloat16 *>(residual), out, ctx.status,
                              static_cast<unsigned long long>(ctx.timeout_ns));
}

}  // namespace

cudaError_t launch_gemm_codes_pair(const void *A16, const void *B16, int64_t M, int64_t N,
                                   int64_t K, const float *sx, const float *sw, const void *bias,
                                   const void *residual, void *out, int out_kind, int pair_n,
                                   const LaunchCtx &ctx) {
    if (M <= 0 || N <= 0) return cudaSuccess;
#define CK_GEMM_PN(PNV)                                                                              \
    if (pair_n == PNV) {                                                                             \
        if (out_kind == kOutS32)                                                                     \
            return launch_pair_t<PNV, kOutS32>(A16, B16, M, N, K, sx, sw, bias, residual, out, ctx); \
        if (out_kind == kOutGlu)                                                                     \
            return launch_pair_t<PNV, kOutGlu>(A16, B16, M, N, K, sx, sw, bias, residual, out, ctx); \
        return launch_pair_t<PNV, kOutBf16>(A16, B16, M, N, K, sx, sw, bias, residual, out, ctx);    \
    }
    CK_GEMM_PN(224)
    CK_GEMM_PN(128)
    CK_GEMM_PN(256)
#undef CK_GEMM_PN
    return cudaErrorInvalidValue;
}

}  // namespace ck
