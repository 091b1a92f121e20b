// gemm_tcgen05.cu -- exact-integer INT8 GEMM on GB300's 5th-generation tensor
// cores, with the ConvRot dequantization fused into the epilogue.
//
//   acc[m, n] = sum_k xq[m, k] * Wq[n, k]                (exact int32)
//   y[m, n]   = bf16( f32(acc) * sx[m] * sw[n] + bias[n] + residual[m, n] )
// comfy-kitchen PR #277, "Summary" / "The key observation": an INT8 x INT8
// GEMM with int32 accumulation, run in the rotated basis and dequantized with
// the per-token and per-output-row scales.
//
// sm_103a has no integer kind for tcgen05.mma, so the codes are multiplied as
// fp16 values (every |q| <= 127 is exact in fp16, every product |p| <= 16129
// is exact in the f32 accumulator).  A sum of at most 1024 products is an
// integer of magnitude at most 1024 * 16129 = 16,516,096 < 2^24, so every
// partial sum is exact in f32 whatever order the tensor core adds in.  The K
// loop is therefore cut into chunks of 1024, the largest power of two under
// that bound (the conversions are costly: going from 512 to 1024 took the
// 4096^3 GEMM from 113 to 101 us on GB300): each
// chunk accumulates into one of two TMEM buffers (alternating), and the
// epilogue warps convert each finished chunk to int32 and add it to per-thread
// int32 sums while the tensor core fills the other buffer.  The int32 result
// is exact for any K.
//
// Structure (persistent: at most one CTA per SM walking output tiles of
// 128 x BN, m fastest, strided by the grid; 10 warps):
//   warp 0     : TMA producer -- A (codes [M, K]) and B (codes [N, K]) tiles of
//                64 K-columns, 128-byte swizzle, into a STAGES-deep ring.
//   warp 1     : TMEM allocator + tcgen05.mma issuer (M=128, N=BN, K=16 per
//                instruction, 4 per stage; the warp walks the ring, one
//                elected lane issues: gemm_issue.cuh).
//   warps 2..9 : epilogue; warp w reads TMEM lanes 32*(w%4) .. +31 (its
//                row quarter) and one half of the BN columns.
// The TMA ring, the MMA chunk counter and the TMEM buffer parity run on across
// tiles, so a tile's dequant and stores (from registers) overlap the next
// tile's MMAs.  Every mbarrier wait is bounded in time (ptx.cuh); a wait that
// runs out makes all roles stop, drain what they have in flight, free TMEM and
// return.
#include <cuda_bf16.h>
#include <stdio.h>

#include <cmath>

#include "gemm_epilogue.cuh"
#include "gemm_issue.cuh"
#include "internal.h"
#include "launch_util.h"
#include "ptx.cuh"

namespace ck {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;                  // one 128-byte swizzle row of fp16
constexpr int kThreads = 320;            // 10 warps
constexpr int kChunkBlocks = 16;         // exact-f32 chunk: 16 x 64 = 1024 products

template <int BN>
struct GemmCfg {
    static constexpr int kStages = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemCols = 2 * BN;  // two accumulator buffers
    static constexpr int kBarBytes = 256;
    // stage ring, barriers, the epilogue's staged scales, alignment slack
    static constexpr size_t kSmemBytes =
        static_cast<size_t>(kStages) * kStageBytes + kBarBytes + ep::staging_bytes(BN) + 1024;
};

template <int BN, int OUT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_codes_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  int M, int N, int K, int m_tiles, const float *__restrict__ sx,
                  const float *__restrict__ sw, const __nv_bfloat16 *__restrict__ bias,
                  const __nv_bfloat16 *residual, void *out, unsigned int *status,
                  unsigned long long timeout_ns) {
    using Cfg = GemmCfg<BN>;
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t smem_s = raw_s + pad;
    // barriers after the stage ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * Cfg::kStageBytes);
    const uint32_t bars_s = smem_s + S * Cfg::kStageBytes;
    auto full_bar = [&](int s) { return bars_s + 8u * s; };
    auto empty_bar = [&](int s) { return bars_s + 8u * (S + s); };
    auto accf_bar = [&](int b) { return bars_s + 8u * (2 * S + b); };
    auto acce_bar = [&](int b) { return bars_s + 8u * (2 * S + 2 + b); };
    const uint32_t done_bar = bars_s + 8u * (2 * S + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *ep_sw = reinterpret_cast<float *>(smem + S * Cfg::kStageBytes + Cfg::kBarBytes);
    float *ep_b = ep_sw + BN;
    auto sA = [&](int s) { return smem_s + s * Cfg::kStageBytes; };
    auto sB = [&](int s) { return smem_s + s * Cfg::kStageBytes + Cfg::kABytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total_tiles = m_tiles * ((N + BN - 1) / BN);
    const int num_kb = K / kBK;
    const int nchunks = (num_kb + kChunkBlocks - 1) / kChunkBlocks;
    const WaitCtl ctl{abort_flag, status, timeout_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 8);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // A kernel queued behind this one may launch now: it waits for our end
    // before it touches anything we read or write.
    pdl_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const int my_tiles =
            static_cast<int>(blockIdx.x) < total_tiles ? (total_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        const int total_kb = my_tiles * num_kb;
        // The weights do not depend on the previous kernel: the first stages'
        // B tiles are requested before waiting on it, A after.
        const int pre = total_kb > 0 ? min(S, num_kb) : 0;
        if (elect_one()) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            for (int kb = 0; kb < pre; ++kb) {
                mbar_arrive_expect_tx(full_bar(kb), Cfg::kStageBytes);
                tma_load_2d(sB(kb), &tmB, full_bar(kb), kb * kBK, (blockIdx.x / m_tiles) * BN);
            }
        }
        __syncwarp();
        pdl_wait();  // A (the activation codes) comes from the previous kernel
        int issued = 0;
        produce_loop<S>(
            total_kb, num_kb, pre, blockIdx.x, gridDim.x, empty_bar(0), ctl,
            [&](int tile, int &a_row, int &b_row) {
                a_row = (tile % m_tiles) * kBM;
                b_row = (tile / m_tiles) * BN;
            },
            [&](int st, int kb, int a_row, int b_row, bool whole) {
                if (whole) {
                    mbar_arrive_expect_tx(full_bar(st), Cfg::kStageBytes);
                    tma_load_2d(sB(st), &tmB, full_bar(st), kb * kBK, b_row);
                }
                tma_load_2d(sA(st), &tmA, full_bar(st), kb * kBK, a_row);
            },
            issued);
        if (*abort_flag && elect_one()) {
            // let the copies still in flight land before the CTA exits
            const int first = issued > S ? issued - S : 0;
            for (int kb = first; kb < issued; ++kb)
                mbar_wait_drain(full_bar(kb % S), (kb / S) & 1, timeout_ns, status);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
        const int my_tiles =
            static_cast<int>(blockIdx.x) < total_tiles ? (total_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        const IssueBars ib{full_bar(0), empty_bar(0), accf_bar(0), acce_bar(0)};
        issue_mma_loop<S, kChunkBlocks, Cfg::kStageBytes / 16>(
            my_tiles * num_kb, num_kb, tmem_base, BN, ib, sdesc_kmajor_sw128(sA(0)),
            sdesc_kmajor_sw128(sB(0)), ctl,
            [](uint32_t d, uint64_t a, uint64_t b, uint32_t acc) { mma_f16_ss(d, a, b, idesc, acc); },
            [](uint32_t bar) { mma_commit(bar); });
        // no MMA may be in flight when TMEM is released (the commit comes from
        // the lane that issued them)
        if (elect_one()) {
            mma_commit(done_bar);
            mbar_wait_drain(done_bar, 0, timeout_ns, status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        constexpr int kCols = BN / 2;
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const int et = threadIdx.x - 64;  // 0..255 over the epilogue warps
        float s_x = 0.f;  // this thread's row scale in the current tile
        if constexpr (OUT != kOutS32) pdl_wait();  // sx comes from the previous kernel
        bool ok = true;
        int gc = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            const int m_tile = tile % m_tiles;
            const int n_tile = tile / m_tiles;
            if constexpr (OUT != kOutS32) {
                ep::sync();  // the previous tile's dequant no longer reads the staging
                if constexpr (OUT == kOutGlu)
                    ep::stage_glu(ep_sw, ep_b, et, BN, n_tile * BN, N, sw, bias);
                else
                    ep::stage(ep_sw, ep_b, et, BN, n_tile * BN, N, sw, bias);
                const int m_row = m_tile * kBM + q * 32 + lane;
                s_x = m_row < M ? sx[m_row] : 0.f;
            }
            int32_t acc[kCols];
#pragma unroll
            for (int i = 0; i < kCols; ++i) acc[i] = 0;
            for (int c = 0; c < nchunks && ok; ++c, ++gc) {
                const int buf = gc & 1;
                // one lane waits, the warp follows: tcgen05.ld below is warp-collective
                int got = 0;
                if (lane == 0) got = mbar_wait(accf_bar(buf), (gc >> 1) & 1, ctl) ? 1 : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(buf * BN + h * kCols);
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
                if (lane == 0) mbar_arrive(acce_bar(buf));
            }
            // the tile's sums are in registers: its stores overlap the next tile's MMAs
            const int n0 = n_tile * BN + h * kCols;
            if constexpr (OUT == kOutS32) {
                if (!ok) break;
                const int m = m_tile * kBM + q * 32 + lane;
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
                    ep::glu_store<kCols>(acc, m_tile * kBM + q * 32, lane, M, n0, N, s_x,
                                         ep_sw + h * kCols, ep_b + h * kCols, static_cast<float *>(out));
                else
                    ep::dequant_store<kCols>(acc, m_tile * kBM + q * 32, lane, M, n0, N, s_x,
                                             ep_sw + h * kCols, ep_b + h * kCols, residual,
                                             static_cast<__nv_bfloat16 *>(out));
            }
        }  // tile loop
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

// Tensor map of an fp16 [rows, K] row-major matrix, box = 64 (K) x box_rows,
// 128-byte swizzle, out-of-range elements read as zero (cached by value).
bool make_map_f16(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows) {
    return tensor_map_2d(map, ptr, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rows, K, kBK, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int BN, int OUT>
cudaError_t launch_bn(const void *A16, const void *B16, int64_t M, int64_t N, int64_t K,
                      const float *sx, const float *sw, const void *bias,
                      const void *residual, void *out, const LaunchCtx &ctx) {
    using Cfg = GemmCfg<BN>;
    CUtensorMap ma, mb;
    if (!make_map_f16(&ma, A16, M, K, kBM) || !make_map_f16(&mb, B16, N, K, BN))
        return cudaErrorInvalidValue;
    auto kern = gemm_codes_kernel<BN, OUT>;
    // the shared-memory opt-in belongs to each device's copy of the kernel
    if (cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                            static_cast<int>(Cfg::kSmemBytes));
        e != cudaSuccess)
        return e;
    const int m_tiles = static_cast<int>((M + kBM - 1) / kBM);
    const int n_tiles = static_cast<int>((N + BN - 1) / BN);
    cudaLaunchConfig_t cfg = {};
    const int sms = sm_count();
    if (sms < 2) return cudaErrorInvalidDevice;
    const int tiles = m_tiles * n_tiles;
    cfg.gridDim = dim3(static_cast<unsigned>(tiles < sms ? tiles : sms));  // persistent
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ctx.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, static_cast<int>(M), static_cast<int>(N),
                              static_cast<int>(K), m_tiles, sx, sw,
                              static_cast<const __nv_bfloat16 *>(bias),
                              static_cast<const __nv_bfloat16 *>(residual), out, ctx.status,
                              static_cast<unsigned long long>(ctx.timeout_ns));
}

// Variant choice: estimated time = rounds of tiles x columns each SM computes
// per tile / the variant's relative throughput (per SM and column, measured on
// GB300).  The wide variants' at 4096 x 3072 -> 24576, where 20-23 rounds leave
// little tile quantization: CTA pairs with 224-column tiles 1.0 (306 us),
// pairs with 256-column tiles 0.97, one-SM 256-wide tiles 0.87.  The narrow
// ones, which win only on problems of a round or two, at one round (1024 x
// 4096 -> 1024): pairs with 128-column tiles 0.71, one-SM 128-wide 0.63,
// 64-wide 0.32 (at 40-80 rounds they fall to 0.60, 0.59, 0.31, and the wide
// ones take those problems anyway).  Returns the tile code of
// set_forced_gemm_bn.
int pick_tile(int64_t M, int64_t N, int num_sms) {
    struct Variant {
        int code, rows, cols;
        double eff;
        bool pair;
    };
    const Variant vs[6] = {{448, 256, 224, 1.0, true},   {512, 256, 256, 0.97, true},
                           {256, 128, 256, 0.87, false}, {2128, 256, 128, 0.71, true},
                           {128, 128, 128, 0.63, false}, {64, 128, 64, 0.32, false}};
    double best = 1e300;
    int choice = 448;
    for (const Variant &v : vs) {
        const double tiles = static_cast<double>((M + v.rows - 1) / v.rows) * ((N + v.cols - 1) / v.cols);
        const double slots = v.pair ? num_sms / 2 : num_sms;
        const double t = std::ceil(tiles / slots) * v.cols / v.eff;
        if (t < best * 0.999) {
            best = t;
            choice = v.code;
        }
    }
    return choice;
}

}  // namespace

// test hook: 0 = automatic, 64/128/256 = one-CTA tile width, 512 / 448 / 2128 =
// CTA pairs with 256- / 224- / 128-column tiles, 4512 = K split between two pairs
static int g_forced_bn = 0;
void set_forced_gemm_bn(int bn) {
    g_forced_bn = (bn == 64 || bn == 128 || bn == 256 || bn == 512 || bn == 448 || bn == 2128 ||
                   bn == 4512)
                      ? bn
                      : 0;
}

// K split between two pairs (one 256 x 256 tile per 4-CTA cluster): measured
// on GB300 as about 10.3 us + 0.278 us per k-block of each half, against
// 7.2 us + 0.195 us per k-block for one round of 256 x 128 pair tiles (the
// fixed part is the exchange of the halves' sums: the last chunk's drain, a
// 64 KB copy between the pairs' shared memories at ~35 GB/s, then the
// dequant).  Taken when every tile has its cluster at once and K >= 6144,
// where that gains >= 9 % (2048 x 1024 <- 12288: 37.0 against 44.7 us; at
// K = 3072 it is 17.0 against 16.6 us).
bool split_k_pays(int64_t M, int64_t N, int64_t K, int sms) {
    const int64_t tiles = ((M + 255) / 256) * ((N + 255) / 256);
    return K >= 6144 && 4 * tiles <= sms;
}

int gemm_tile_choice(int64_t M, int64_t N, int64_t K, int sms) {
    if (g_forced_bn) return g_forced_bn;
    if (split_k_pays(M, N, K, sms)) return 4512;
    // One chunk of K (<= 1024) leaves every tile's fixed costs exposed: up to
    // two rounds of them 128 x 128 one-SM tiles are as good as any; beyond,
    // the pairs win (measured on GB300: 2048 x 1024 -> 3072, 2.5 rounds:
    // 224-column pairs 17.9 us, one-SM 128 18.6, 128-column pairs 18.7,
    // one-SM 256 18.9, 256-column pairs 19.5).
    const bool short_k =
        K <= 1024 && ((M + kBM - 1) / kBM) * ((N + 127) / 128) <= 2 * static_cast<int64_t>(sms);
    return short_k ? 128 : pick_tile(M, N, sms);
}

cudaError_t launch_gemm_codes(const void *A16, const void *B16, int64_t M, int64_t N, int64_t K,
                              const float *sx, const float *sw, const void *bias,
                              const void *residual, void *out, int out_kind, const LaunchCtx &ctx) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (out_kind != kOutBf16 && out_kind != kOutS32 && out_kind != kOutGlu) return cudaErrorInvalidValue;
    const int sms = sm_count();
    if (sms < 2) return cudaErrorInvalidDevice;
    int bn = gemm_tile_choice(M, N, K, sms);
    if (bn == 4512) {
        // the automatic choice also needs every tile's cluster resident at once
        const int64_t tiles = ((M + 255) / 256) * ((N + 255) / 256);
        if (out_kind != kOutGlu && K / 64 >= 2 &&
            (g_forced_bn == 4512 || tiles <= splitk_resident_clusters()))
            return launch_gemm_codes_splitk(A16, B16, M, N, K, sx, sw, bias, residual, out, out_kind, ctx);
        bn = pick_tile(M, N, sms);
    }
    if (bn >= 448)
        return launch_gemm_codes_pair(A16, B16, M, N, K, sx, sw, bias, residual, out, out_kind,
                                      bn == 2128 ? 128 : bn / 2, ctx);
#define CK_GEMM_BN(BNV)                                                                          \
    if (bn == BNV) {                                                                             \
        if (out_kind == kOutS32)                                                                 \
            return launch_bn<BNV, kOutS32>(A16, B16, M, N, K, sx, sw, bias, residual, out, ctx); \
        if (out_kind == kOutGlu)                                                                 \
            return launch_bn<BNV, kOutGlu>(A16, B16, M, N, K, sx, sw, bias, residual, out, ctx); \
        return launch_bn<BNV, kOutBf16>(A16, B16, M, N, K, sx, sw, bias, residual, out, ctx);    \
    }
    CK_GEMM_BN(256)
    CK_GEMM_BN(128)
    CK_GEMM_BN(64)
#undef CK_GEMM_BN
    return cudaErrorInvalidValue;
}

}  // namespace ck
