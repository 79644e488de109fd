// Deterministic backward: the order in which a dQ tile takes its key blocks'
// contributions. Shared by the d <= 128 kernel (bwd.cu) and the d = 192 / 256
// kernel (bwd_wide.cu); `Tile` is either one's work tile (fields b, n, lq, lk,
// q_row0, mcol). Query and key blocks are 128 rows.
//
// Each dQ tile (b, h, m) has a semaphore counting the key blocks that have
// added their contribution (two in the wide kernel, one per dQ column chunk).
// A key block waits until the count equals the number of blocks ahead of it,
// adds its contribution, waits for the adds to complete and increments the
// count: the sum is taken in the same order on every run (FlashAttention-4
// paper, Section 3.2.4). The functions are also compiled for the host, where
// tests/sched_host.cu checks that the turns of every dQ tile's contributors
// are 0, 1, ..., K - 1 (a gap or a repeat would leave a block waiting).
#pragma once

#include "kernels.h"
#include "mask.cuh"

namespace attn {

// Index of dQ tile (b, h, m) among the semaphores (dense: [B, H, nq]; varlen:
// per head, sequence b's blocks from q_row0 / 128 + b on, which leaves room for
// every sequence's ragged last block).
template <class Tile>
__host__ __device__ __forceinline__ long dq_semaphore(const BwdParams& p, const Tile& f, int h, int m, bool varlen) {
    const Geometry& g = p.g;
    return varlen ? (long)h * (g.Lq / 128 + g.B + 1) + f.q_row0 / 128 + f.b + m : ((long)f.b * g.H + h) * p.nq + m;
}

// The number of key blocks that go before block f.n at query block m of head
// h. Order: from the highest key block down with a right mask bound (shortest
// tiles first, so no tile waits at its first dQ write), else ascending. The key
// blocks that see query block m form one range [n_lo, n_hi) (the mask band);
// with a block mask only the kept ones count.
template <bool kBand, bool kSparse, class Tile>
__host__ __device__ __forceinline__ int dq_turn(const BwdParams& p, const Tile& f, int h, int m) {
    const Geometry& g = p.g;
    int n_lo, n_hi;
    band_key_blocks(mask_band(f.lq, f.lk, g.win_left, g.win_right), m * 128, m * 128 + 127, 128, &n_lo, &n_hi);
    const bool spt = g.causal != 0;
    int before = spt ? n_hi - 1 - f.n : f.n - (kBand ? n_lo : 0);
    if (kSparse && f.mcol) {
        const unsigned char* row =
            p.mask.ptr + ((p.mask.heads == 1 ? 0 : (long)h) * mask_rows(g) + m) * mask_cols(g);
        before = 0;
        for (int x = spt ? f.n + 1 : n_lo; x < (spt ? n_hi : f.n); ++x) before += row[x] != 0;
    }
    return before;
}

}  // namespace attn
