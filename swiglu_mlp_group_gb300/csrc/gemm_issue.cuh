// gemm_issue.cuh -- the TMA producer and the MMA issuer of the tcgen05 GEMMs
// (one-SM and CTA-pair kernels).  Each is one warp walking the CTA's k-blocks
// (its tiles x K / 64, tile after tile) around the ring of S stages: the
// producer refills a stage once the MMAs have released it; the issuer runs,
// per k-block, the four K = 16 MMAs of the stage, releases it and, at the end
// of each 1024-product chunk, publishes the accumulator buffer.
//
// Shape of the loop (timed in isolation on GB300, ns per k-block of four MMAs,
// by a diagnostic kernel that ran the issue loop alone on zero operands):
// keeping the stage index and the round's parity at run time in one lane of
// the warp costs ~260 ns per k-block whatever the tile width -- twice the
// MMAs' own 132 ns at N = 128, 13 % over their 230 ns at N = 224.  Walking
// the ring in rounds of S k-blocks with the stage index a compile-time
// constant in each unrolled step (barrier address and descriptors =
// loop-invariant base + constant), the whole warp running the loop and one
// elected lane issuing, it takes 142 / 230 / 263 ns at N = 128 / 224 / 256
// (the last two the MMAs' own time).  The producer walks the ring the same way.
#pragma once

#include "ptx.cuh"

namespace ck {

// Barrier addresses: full[s] = full0 + 8 s, empty[s] = empty0 + 8 s,
// accf[b] = accf0 + 8 b, acce[b] = acce0 + 8 b (b = TMEM accumulator buffer).
struct IssueBars {
    uint32_t full0, empty0, accf0, acce0;
};

// Runs in every lane of the issuing warp.  total_kb = tiles of this CTA x
// num_kb.  mma(d_tmem, adesc, bdesc, accumulate) and commit(bar) issue one
// tcgen05 instruction each (called from one lane).  Returns false when a wait
// gave up (the CTA's abort flag is then set); nothing is issued after that.
template <int S, int kChunkBlocks, uint32_t kStageDescStep, typename Mma, typename Commit>
__device__ __forceinline__ bool issue_mma_loop(int total_kb, int num_kb, uint32_t tmem_base,
                                               uint32_t buf_cols, const IssueBars &bars,
                                               uint64_t adesc0, uint64_t bdesc0, const WaitCtl &ctl,
                                               Mma mma, Commit commit) {
    uint32_t ph = 0;     // parity of the ring's current round
    int kb = 0;          // k-block within the tile
    int gc = 0;          // accumulator chunk counter (TMEM buffer = gc % 2)
    int buf = 0;
    uint32_t d_tmem = tmem_base;
    for (int g0 = 0; g0 < total_kb; g0 += S) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            if (g0 + s >= total_kb) break;
            const bool first = kb % kChunkBlocks == 0;
            if (first) {
                buf = gc & 1;
                // the epilogue has drained what this buffer held two chunks ago
                if (gc >= 2 &&
                    !__all_sync(0xffffffffu, mbar_wait(bars.acce0 + 8u * buf, ((gc >> 1) - 1) & 1, ctl)))
                    return false;
                tc_fence_after_sync();
                d_tmem = tmem_base + static_cast<uint32_t>(buf) * buf_cols;
            }
            if (!__all_sync(0xffffffffu, mbar_wait(bars.full0 + 8u * s, ph, ctl))) return false;
            tc_fence_after_sync();
            const bool last = kb + 1 == num_kb || (kb + 1) % kChunkBlocks == 0;
            if (elect_one()) {
                // the address field of a descriptor is (address >> 4): stage s of
                // the ring is the base plus a constant
                const uint64_t ad = adesc0 + static_cast<uint64_t>(s) * kStageDescStep;
                const uint64_t bd = bdesc0 + static_cast<uint64_t>(s) * kStageDescStep;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma(d_tmem, ad + 2u * k, bd + 2u * k, (!first || k > 0) ? 1u : 0u);
                commit(bars.empty0 + 8u * s);
                if (last) commit(bars.accf0 + 8u * buf);
            }
            __syncwarp();
            if (last) ++gc;
            if (++kb == num_kb) kb = 0;
        }
        ph ^= 1u;
    }
    return true;
}

// Runs in every lane of the producer warp.  The first `pre` k-blocks (pre <= S)
// had their stage armed and their B tile requested before the kernel waited
// on its predecessor: for those only A is loaded.  tile_rows(tile, a_row,
// b_row) gives a tile's operand rows; issue(s, kb, a_row, b_row, whole) loads
// stage s for k-block kb (whole: arm the stage and load A and B; else A only;
// called from one lane).  `issued` = k-blocks requested.  Returns false when a
// wait gave up.
template <int S, typename TileRows, typename Issue>
__device__ __forceinline__ bool produce_loop(int total_kb, int num_kb, int pre, int first_tile,
                                             int tile_step, uint32_t empty0, const WaitCtl &ctl,
                                             TileRows tile_rows, Issue issue, int &issued) {
    uint32_t ph = 0;
    int kb = 0;
    int tile = first_tile;
    int a_row = 0, b_row = 0;
    tile_rows(tile, a_row, b_row);
    issued = 0;
    for (int g0 = 0; g0 < total_kb; g0 += S) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int g = g0 + s;
            if (g >= total_kb) break;
            const bool whole = g >= pre;
            // the MMAs have read what this stage held one round ago
            if (whole && !__all_sync(0xffffffffu, mbar_wait(empty0 + 8u * s, ph ^ 1u, ctl)))
                return false;
            if (elect_one()) issue(s, kb, a_row, b_row, whole);
            __syncwarp();
            issued = g + 1;
            if (++kb == num_kb) {
                kb = 0;
                tile += tile_step;
                tile_rows(tile, a_row, b_row);
            }
        }
        ph ^= 1u;
    }
    return true;
}

}  // namespace ck
