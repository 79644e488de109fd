// Persistent tile scheduling: longest-processing-time-first (LPT) orders.
//
// FlashAttention-4 paper, Section 3.3 "Scheduling":
//  * causal LPT: the batch is the outermost dimension; heads are split into
//    sections whose K/V fit in L2; within a section the scheduler walks the
//    m-blocks in reverse (longest causal rows first), and within an m-block
//    the heads of the section;
//  * varlen LPT: sequences are sorted by the cost of their longest work tile
//    (descending) into a virtual-to-real batch map that the kernel walks. The
//    forward's tiles cover query rows and the longest visits every key, so it
//    sorts by key count; the backward's cover keys and sorts by query count
//    (the same order when queries and keys share their offsets).
// Blog post on FA4 (qian.cx), "StaticPersistentTileScheduler": at most one
// CTA per SM; CTA c takes tiles c, c + grid, c + 2*grid, ...
//
// A work tile is (b, h, m) where m indexes a block of query rows (forward:
// a pair of 128-row Q tiles; backward: one 128-row K/V block). The same
// closed-form walk is used for dense problems; varlen problems walk the
// sorted sequence map built in shared memory by sched_varlen_build().
#pragma once

#include <cstdint>

namespace attn {

// The index functions below are also compiled for the host, where
// tests/test_sched.py checks their coverage and balance.

constexpr int kMaxVarlenBatch = 1024;   // sequences per varlen call (shared-memory map)

struct Tile {
    int b, h, m;   // batch (real sequence index), head, row-block index
};

// Walk position `rem` inside one batch entry with `nm` row blocks and H heads,
// heads grouped `hs` at a time; `reverse` walks row blocks from the last.
__host__ __device__ __forceinline__ void sched_within_batch(int rem, int nm, int H, int hs, bool reverse,
                                                   int& h, int& m) {
    int s = rem / (hs * nm);
    int h0 = s * hs;
    const int sec_h = hs < H - h0 ? hs : H - h0;
    int idx = rem - s * hs * nm;
    int mi = idx / sec_h;
    h = h0 + (idx - mi * sec_h);
    m = reverse ? nm - 1 - mi : mi;
}

// The k-th work tile of CTA `cta` among `grid` persistent CTAs. Tiles are
// handed out in rounds of `grid`, alternating direction every round
// (boustrophedon), so that with tiles ordered longest first the per-CTA sums
// of tile lengths stay balanced: for causal problems a plain round-robin left
// the busiest CTA with 17-23% more work than the mean, this order with under
// 2% (host simulation of the 4096- and 8192-row workloads). Increasing in k,
// so each CTA walks its tiles in increasing index order.
__host__ __device__ __forceinline__ int snake_tile(int cta, int k, int grid) {
    return k * grid + ((k & 1) ? grid - 1 - cta : cta);
}

// Dense causal problems: every (batch, head) has the same row-block lengths,
// so the global longest-first order is by row-block level, then batch, then
// head. m_desc: a larger row-block index is the longer tile (forward). For
// non-causal problems all tiles are equally long and the L2-section order
// below is kept (it measured ~2% faster there).
__host__ __device__ __forceinline__ Tile sched_dense_lpt(int t, int B, int H, int nm, bool m_desc) {
    Tile ti;
    const int level = t / (B * H);
    const int rem = t - level * (B * H);
    ti.b = rem / H;
    ti.h = rem - ti.b * H;
    ti.m = m_desc ? nm - 1 - level : level;
    return ti;
}

__host__ __device__ __forceinline__ Tile sched_dense(int t, int H, int nm, int hs, bool reverse) {
    Tile ti;
    int per_b = H * nm;
    ti.b = t / per_b;
    sched_within_batch(t - ti.b * per_b, nm, H, hs, reverse, ti.h, ti.m);
    return ti;
}

// Whether a causal dense backward (default mode) should walk its heads in
// L2-sized sections (sched_dense) rather than in one global longest-first order
// (sched_dense_lpt). Sections keep a section's Q, dO and dQ accumulator in L2;
// their tile lengths form a sawtooth (longest first within each section), which
// the boustrophedon hand-out balances less well. Measured on GB300 (d = 128
// unless stated): B1 H32 L32768 gained 10% (a 537 MB working set of Q and dO,
// 7% imbalance), B4 H16 L4096 11% (134 MB, 4%), B2 H16 L8192 lost 2% (134 MB,
// 10.5%; d = 64 lost 11%). So: sections when the heads' Q and dO exceed three
// L2s, or when the sectioned order leaves the busiest CTA under 5% above the
// mean (host simulation of the hand-out below). units: key blocks (or pairs)
// per (b, h); nkv: key/value heads; split: tiles per key block; grid: CTAs (or
// clusters) of the launch; ws_bytes: Q and dO bytes of all query heads.
inline bool sched_sections_pay(int B, int nkv, int units, int hs, int split, int grid, double ws_bytes) {
    if (ws_bytes > 3.0 * 129.0e6) return true;
    const long n = (long)B * nkv * units * split;
    if (grid <= 0 || n <= grid || hs >= nkv * B) return false;
    double total = 0, worst = 0;
    for (int cta = 0; cta < grid; ++cta) {
        double load = 0;
        for (int k = 0;; ++k) {
            const int t = snake_tile(cta, k, grid);
            if (t >= n) break;
            // tile t of the sectioned order: the key block's level inside its section
            const int u = t / split;
            const int per_b = nkv * units;
            const int rem = u % per_b;
            const int s = rem / (hs * units), h0 = s * hs;
            const int sec_h = hs < nkv - h0 ? hs : nkv - h0;
            const int level = (rem - s * hs * units) / sec_h;
            load += units - level;   // causal: the key block at level l sees units - l query blocks
        }
        total += load;
        worst = load > worst ? load : worst;
    }
    return worst < 1.05 * total / grid;
}

// Tables for a varlen problem (shared memory in the forward, the workspace in
// the backward).
struct VarlenMap {
    int start[kMaxVarlenBatch + 1];     // query offsets (cu_seqlens copy)
    int start_k[kMaxVarlenBatch + 1];   // key offsets (cu_seqlens_k, or cu_seqlens again)
    int order[kMaxVarlenBatch];         // virtual -> real sequence (longest first)
    int pre[kMaxVarlenBatch + 1];       // prefix count of tiles in virtual order
};

__host__ __device__ __forceinline__ int vm_lq(const VarlenMap& vm, int b) { return vm.start[b + 1] - vm.start[b]; }
__host__ __device__ __forceinline__ int vm_lk(const VarlenMap& vm, int b) { return vm.start_k[b + 1] - vm.start_k[b]; }

// Build the map with all `nthreads` threads of the calling CTA (every thread
// of it must call); ends with __syncthreads. over_keys = false: work tiles
// cover query rows (forward), a sequence has heads * ceil(Lq / rows_per_block)
// of them and sorts by Lk; over_keys = true: tiles cover keys (backward),
// heads * ceil(Lk / rows_per_block), sorted by Lq. Ties: the other length,
// then the sequence index.
__device__ __forceinline__ void sched_varlen_build(VarlenMap& vm, const int* cu, const int* cu_k, int B,
                                                   int heads, int rows_per_block, bool over_keys, int tid,
                                                   int nthreads) {
    for (int i = tid; i <= B; i += nthreads) {
        vm.start[i] = cu[i];
        vm.start_k[i] = cu_k[i];
    }
    __syncthreads();
    for (int i = tid; i < B; i += nthreads) {
        const int ki = over_keys ? vm_lq(vm, i) : vm_lk(vm, i), oi = over_keys ? vm_lk(vm, i) : vm_lq(vm, i);
        int rank = 0;
        for (int j = 0; j < B; ++j) {
            const int kj = over_keys ? vm_lq(vm, j) : vm_lk(vm, j), oj = over_keys ? vm_lk(vm, j) : vm_lq(vm, j);
            rank += (kj > ki) || (kj == ki && (oj > oi || (oj == oi && j < i)));
        }
        vm.order[rank] = i;
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int k = 0; k < B; ++k) {
            vm.pre[k] = acc;
            const int b = vm.order[k];
            const int L = over_keys ? vm_lk(vm, b) : vm_lq(vm, b);
            acc += heads * ((L + rows_per_block - 1) / rows_per_block);
        }
        vm.pre[B] = acc;
    }
    __syncthreads();
}

// over_keys as in sched_varlen_build: the tile's row blocks split Lk, else Lq.
__host__ __device__ __forceinline__ Tile sched_varlen(const VarlenMap& vm, int t, int B, int H, int rows_per_block,
                                             int hs, bool reverse, bool over_keys) {
    int lo = 0, hi = B - 1;   // largest k with pre[k] <= t
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (vm.pre[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    Tile ti;
    ti.b = vm.order[lo];
    const int L = over_keys ? vm_lk(vm, ti.b) : vm_lq(vm, ti.b);
    const int nm = (L + rows_per_block - 1) / rows_per_block;
    sched_within_batch(t - vm.pre[lo], nm, H, hs, reverse, ti.h, ti.m);
    return ti;
}

}  // namespace attn
