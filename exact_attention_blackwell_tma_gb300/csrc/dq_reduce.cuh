// dQ accumulation: each dQ warp adds its own 32 query rows of a dQ tile to the
// fp32 accumulator (FlashAttention-4 paper, Section 3.2.2: dQ is accumulated in
// global memory across the key blocks that see a query block).
//
// A warp stages its rows through its own 4 KB of each 32-column box of the
// stage tile (rows 32 w .. 32 w + 31 of a 128-row swizzled tile) and its lane 0
// issues TMA reduce-adds of 32-row x 32-column boxes as soon as the warp has
// written them: no warpgroup barrier and no single issuing thread, so the four
// warps keep four streams of reduce-adds in flight (with one thread issuing
// 128-row boxes for the whole warpgroup the backward step was bound by this
// path: B1 H32 L32768 d128 non-causal 920 -> 1100 TF/s on GB300).
#pragma once

#include "ptx.cuh"

namespace attn {

// Stage and add `rounds` x 64 columns of this thread's query row (row[], fp32
// bits, rounds <= 2): round r covers accumulator columns col0 + 64 r .. + 63.
// stage / stage_s: the 128-row stage tile (two 16 KB boxes of 32 columns),
// generic and shared-window addresses; quarter: this warp's row quarter;
// rq = 32 quarter + lane. Returns after lane 0 has committed the last round;
// the caller then waits for the reads (or the completion) of its own groups.
__device__ __forceinline__ void dq_warp_reduce(const CUtensorMap* tm32, uint8_t* stage, uint32_t stage_s,
                                               const uint32_t* row, int rounds, int col0, int head, int row0,
                                               int quarter, int lane) {
    const int rq = quarter * 32 + lane;
    const uint32_t wbase = stage_s + (uint32_t)quarter * 4096u;
#pragma unroll
    for (int rnd = 0; rnd < 2; ++rnd) {
        if (rnd >= rounds) break;
        if (rnd > 0) {   // this warp's rows of the stage have been read by the previous round
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
        }
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            uint8_t* srow = stage + c2 * 16384 + (rq >> 3) * 1024 + (rq & 7) * 128;
            const int c0 = rnd * 64 + c2 * 32;
#pragma unroll
            for (int j = 0; j < 8; ++j)   // 128-byte swizzle: chunk j at j ^ (row % 8)
                *reinterpret_cast<uint4*>(srow + ((j ^ (rq & 7)) << 4)) =
                    make_uint4(row[c0 + 4 * j], row[c0 + 4 * j + 1], row[c0 + 4 * j + 2], row[c0 + 4 * j + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            // rows past the query block's sequence carry exact zeros (P = 0 there)
            for (int c2 = 0; c2 < 2; ++c2)
                tma_reduce_add_3d(tm32, wbase + c2 * 16384, col0 + rnd * 64 + c2 * 32, head, row0 + quarter * 32);
            bulk_commit_group();
        }
    }
}

}  // namespace attn
