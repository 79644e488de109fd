// Host-side checks of the persistent tile scheduler (csrc/sched.cuh), of
// the mask band's index arithmetic (csrc/mask.cuh) and of the deterministic
// backward's dQ order (csrc/dq_order.cuh), compiled
// by tests/test_sched.py with nvcc and run without a GPU. The index functions
// under test are the ones the kernels call. Prints "OK" and exits 0 when every
// check passes; otherwise prints the first failure and exits 1.
#include <cstdio>
#include <cstdlib>
#include <set>
#include <tuple>
#include <vector>
#include <algorithm>

#include "mask.cuh"
#include "sched.cuh"
#include "dq_order.cuh"

using namespace attn;

static int fail(const char* what, int a, int b, int c) {
    std::printf("FAIL %s (%d %d %d)\n", what, a, b, c);
    std::exit(1);
}

// every tile index in [0, n) is handed to exactly one CTA, each CTA's
// sequence increases (the kernels' loop condition relies on it)
static void check_snake(int n, int grid) {
    std::vector<int> seen(n, 0);
    for (int c = 0; c < grid; ++c) {
        int prev = -1;
        for (int k = 0;; ++k) {
            const int t = snake_tile(c, k, grid);
            if (t >= n) break;
            if (t <= prev) fail("snake not increasing", c, k, t);
            prev = t;
            ++seen[t];
        }
    }
    for (int t = 0; t < n; ++t)
        if (seen[t] != 1) fail("snake coverage", n, grid, t);
}

// the dense walks enumerate every (b, h, m) exactly once
static void check_dense(int B, int H, int nm, int hs) {
    for (int mode = 0; mode < 4; ++mode) {
        std::set<std::tuple<int, int, int>> got;
        int prev_m = -1;
        for (int t = 0; t < B * H * nm; ++t) {
            Tile ti = mode < 2 ? sched_dense(t, H, nm, hs, mode == 1) : sched_dense_lpt(t, B, H, nm, mode == 3);
            if (ti.b < 0 || ti.b >= B || ti.h < 0 || ti.h >= H || ti.m < 0 || ti.m >= nm)
                fail("dense tile out of range", B, H, t);
            got.insert({ti.b, ti.h, ti.m});
            if (mode >= 2) {   // longest first: the row-block level moves monotonically
                const int level = mode == 3 ? nm - 1 - ti.m : ti.m;
                if (level < prev_m) fail("lpt order", B, H, t);
                prev_m = level;
            }
        }
        if ((int)got.size() != B * H * nm) fail("dense coverage", B, H, nm);
    }
}

// a varlen map as the device builds it: tiles split the query rows (forward)
// or the keys (over_keys, backward); sequences sorted by the other length,
// longest first (ties: the tiled length, then the index); prefix counts of
// H * ceil(tiled length / rows) tiles
static void build_map(VarlenMap& vm, const std::vector<int>& lq, const std::vector<int>& lk, int H, int rows,
                      bool over_keys) {
    const int B = (int)lq.size();
    vm.start[0] = vm.start_k[0] = 0;
    for (int i = 0; i < B; ++i) {
        vm.start[i + 1] = vm.start[i] + lq[i];
        vm.start_k[i + 1] = vm.start_k[i] + lk[i];
    }
    const std::vector<int>& key = over_keys ? lq : lk;
    const std::vector<int>& tiled = over_keys ? lk : lq;
    std::vector<int> idx(B);
    for (int i = 0; i < B; ++i) idx[i] = i;
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) {
        return key[a] != key[b] ? key[a] > key[b] : tiled[a] > tiled[b];
    });
    int acc = 0;
    for (int k = 0; k < B; ++k) {
        vm.order[k] = idx[k];
        vm.pre[k] = acc;
        acc += H * ((tiled[idx[k]] + rows - 1) / rows);
    }
    vm.pre[B] = acc;
}

static void check_varlen(const std::vector<int>& lq, const std::vector<int>& lk, int H, int rows, int hs,
                         bool over_keys) {
    static VarlenMap vm;
    build_map(vm, lq, lk, H, rows, over_keys);
    const int B = (int)lq.size(), n = vm.pre[B];
    const std::vector<int>& key = over_keys ? lq : lk;
    const std::vector<int>& tiled = over_keys ? lk : lq;
    std::set<std::tuple<int, int, int>> got;
    int prev_len = 1 << 30;
    for (int t = 0; t < n; ++t) {
        Tile ti = sched_varlen(vm, t, B, H, rows, hs, true, over_keys);
        const int L = tiled[ti.b], nm = (L + rows - 1) / rows;
        if (ti.h < 0 || ti.h >= H || ti.m < 0 || ti.m >= nm) fail("varlen tile out of range", ti.b, ti.h, ti.m);
        if (key[ti.b] > prev_len) fail("varlen not longest first", t, key[ti.b], prev_len);
        prev_len = key[ti.b];
        got.insert({ti.b, ti.h, ti.m});
    }
    int expect = 0;
    for (int L : tiled) expect += H * ((L + rows - 1) / rows);
    if ((int)got.size() != expect || n != expect) fail("varlen coverage", n, expect, (int)got.size());
}

static void check_varlen(const std::vector<int>& lens, int H, int rows, int hs) {
    check_varlen(lens, lens, H, rows, hs, false);
    check_varlen(lens, lens, H, rows, hs, true);
}

// causal balance: per-CTA sums of tile lengths under the longest-first order
// and the boustrophedon hand-out stay within `tol` of the mean
static void check_causal_balance(int B, int H, int L, int rows, bool fwd, int grid, double tol) {
    const int nm = (L + rows - 1) / rows, n = B * H * nm;
    std::vector<double> work(grid, 0.0);
    for (int c = 0; c < grid; ++c)
        for (int k = 0;; ++k) {
            const int t = snake_tile(c, k, grid);
            if (t >= n) break;
            Tile ti = sched_dense_lpt(t, B, H, nm, fwd);
            // forward: row block m sees (m+1)*rows keys; backward: key block m is
            // seen by the query rows from m*rows to L
            work[c] += fwd ? (double)(ti.m + 1) : (double)(nm - ti.m);
        }
    double mx = 0, sum = 0;
    for (double w : work) {
        mx = std::max(mx, w);
        sum += w;
    }
    const double mean = sum / grid;
    if (mx > mean * (1.0 + tol)) fail("causal imbalance (max/mean in percent)", (int)(100 * mx / mean), L, fwd);
}

// mask.cuh against a scan of the mask: per row and per key the range of
// partners, and for groups of rows (keys) the blocks of keys (rows) they reach
static void check_band(int lq, int lk, int wl, int wr) {
    const MaskBand m = mask_band(lq, lk, wl, wr);
    auto seen = [&](int i, int j) {   // query i sees key j: the definition, scanned
        const int d = lk - lq;
        if (j < 0 || j >= lk) return false;
        if (wr >= 0 && j > i + d + wr) return false;
        if (wl >= 0 && j < i + d - wl) return false;
        return true;
    };
    for (int i = 0; i < lq; ++i) {
        const int lo = band_key_lo(m, i), hi = band_key_hi(m, i);
        for (int j = 0; j < lk; ++j)
            if (seen(i, j) != (j >= lo && j < hi)) fail("band key range", i, j, wl * 1000 + wr);
    }
    for (int j = 0; j < lk; ++j) {
        const int lo = band_query_lo(m, j), hi = band_query_hi(m, j);
        for (int i = 0; i < lq; ++i)
            if (seen(i, j) != (i >= lo && i < hi)) fail("band query range", i, j, wl * 1000 + wr);
    }
    for (int span : {128, 256})
        for (int r0 = 0; r0 < lq + 256; r0 += 128) {
            std::vector<char> blk((lk + 127) / 128 + 1, 0);
            for (int i = r0; i < r0 + span && i < lq; ++i)
                for (int j = 0; j < lk; ++j)
                    if (seen(i, j)) blk[j / 128] = 1;
            int jlo, jhi;
            const bool any = band_key_blocks(m, r0, r0 + span - 1, 128, &jlo, &jhi);
            for (int b = 0; b < (int)blk.size(); ++b)
                if ((bool)blk[b] != (any && b >= jlo && b < jhi)) fail("band key blocks", r0, b, wl * 1000 + wr);
        }
    for (int k0 = 0; k0 < lk + 128; k0 += 128) {
        std::vector<char> blk((lq + 127) / 128 + 1, 0);
        for (int j = k0; j < k0 + 128 && j < lk; ++j)
            for (int i = 0; i < lq; ++i)
                if (seen(i, j)) blk[i / 128] = 1;
        int mlo, mhi;
        const bool any = band_query_blocks(m, k0, k0 + 127, 128, &mlo, &mhi);
        for (int b = 0; b < (int)blk.size(); ++b)
            if ((bool)blk[b] != (any && b >= mlo && b < mhi)) fail("band query blocks", k0, b, wl * 1000 + wr);
    }
}


// The deterministic backward's dQ order (dq_order.cuh): for every dQ tile, the
// key blocks that contribute to it -- those whose rows see some row of the
// query block (a scan of the mask) and, with a block mask, whose block it
// keeps -- get the turns 0, 1, ..., K - 1, each once. kBand = false is the
// instantiation for no mask and the causal one.
struct HostTile {
    int b, n, lq, lk, q_row0;
    const unsigned char* mcol;
};

template <bool kBand, bool kSparse>
static void check_dq_turns(int lq, int lk, int wl, int wr, const std::vector<unsigned char>* mask) {
    BwdParams p{};
    p.g.B = 1;
    p.g.H = p.g.Hkv = p.g.group = 1;
    p.g.Lq = lq;
    p.g.Lk = lk;
    p.g.causal = wr >= 0;
    p.g.win_left = wl;
    p.g.win_right = wr;
    p.nq = (lq + 127) / 128;
    p.mask = BlockMask{mask ? mask->data() : nullptr, 1};
    const int nq = (lq + 127) / 128, nk = (lk + 127) / 128;
    auto sees = [&](int i, int j) {
        const int d = lk - lq;
        return !(wr >= 0 && j > i + d + wr) && !(wl >= 0 && j < i + d - wl);
    };
    for (int m = 0; m < nq; ++m) {
        std::vector<int> turns;
        for (int n = 0; n < nk; ++n) {
            bool any = false;
            for (int i = m * 128; i < std::min(lq, m * 128 + 128) && !any; ++i)
                for (int j = n * 128; j < std::min(lk, n * 128 + 128) && !any; ++j) any = sees(i, j);
            if (mask && !(*mask)[(size_t)m * nk + n]) any = false;
            if (!any) continue;
            const HostTile f{0, n, lq, lk, 0, mask ? mask->data() + n : nullptr};
            turns.push_back(dq_turn<kBand, kSparse>(p, f, 0, m));
            if (dq_semaphore(p, f, 0, m, false) != m) fail("dq semaphore index", lq, lk, m);
        }
        std::sort(turns.begin(), turns.end());
        for (int k = 0; k < (int)turns.size(); ++k)
            if (turns[k] != k) fail("dq turns not 0..K-1", m, k, wl * 100000 + wr * 100 + lq % 100);
    }
}

// Every dQ semaphore the kernels address lies inside the array the host
// sizes (bwd_semaphore_count): dense and packed layouts, including the wide
// kernel's second column chunk (index 2 * tile + 1). Distinct dQ tiles get
// distinct semaphores.
static void check_dq_semaphore_bounds(const std::vector<int>& lens, int H, bool varlen) {
    BwdParams p{};
    const int B = (int)lens.size();
    int T = 0;
    for (int L : lens) T += L;
    const int Lq = varlen ? T : lens[0];
    p.g.B = B;
    p.g.H = H;
    p.g.Lq = Lq;
    p.nq = (Lq + 127) / 128;
    const long count = bwd_semaphore_count(B, H, Lq, varlen);
    std::set<long> seen;
    int row0 = 0;
    for (int b = 0; b < B; ++b) {
        const int lq = varlen ? lens[b] : Lq;
        const HostTile f{b, 0, lq, lq, varlen ? row0 : b * Lq, nullptr};
        for (int h = 0; h < H; ++h)
            for (int m = 0; m < (lq + 127) / 128; ++m) {
                const long idx = dq_semaphore(p, f, h, m, varlen);
                if (idx < 0 || 2 * idx + 1 >= count) fail("dq semaphore out of range", b, h, m);
                if (!seen.insert(idx).second) fail("dq semaphore shared", b, h, m);
            }
        row0 += lq;
    }
}

static void check_dq_order() {
    unsigned seed = 12345;
    for (int lq : {1, 130, 300, 517, 1000})
        for (int lk : {1, 130, 300, 517, 1000}) {
            check_dq_turns<false, false>(lq, lk, -1, -1, nullptr);
            check_dq_turns<false, false>(lq, lk, -1, 0, nullptr);
            for (int wl : {-1, 0, 3, 128, 200})
                for (int wr : {-1, 0, 3, 128, 200}) {
                    check_dq_turns<true, false>(lq, lk, wl, wr, nullptr);
                    const int nq = (lq + 127) / 128, nk = (lk + 127) / 128;
                    std::vector<unsigned char> mask((size_t)nq * nk);
                    for (auto& x : mask) {
                        seed = seed * 1103515245u + 12345u;
                        x = (seed >> 16) % 3 != 0;
                    }
                    check_dq_turns<true, true>(lq, lk, wl, wr, &mask);
                }
        }
}

// The backward's choice of tile order for causal dense problems
// (sched_sections_pay) on the benchmark's workloads, as measured on GB300:
// sections for B4 H16 L4096 and B1 H32 L32768, one global order for B2 H16
// L8192 (d = 64 and 128); never sections when every tile fits one round.
static void check_sections_choice() {
    auto ws = [](double B, double H, double L, double d) { return 4.0 * B * L * H * d; };
    if (!sched_sections_pay(4, 16, 32, 16, 1, 152, ws(4, 16, 4096, 128))) fail("sections B4 H16 L4096", 4, 16, 4096);
    if (!sched_sections_pay(1, 32, 256, 3, 1, 152, ws(1, 32, 32768, 128))) fail("sections B1 H32 L32768", 1, 32, 32768);
    if (sched_sections_pay(2, 16, 64, 16, 1, 152, ws(2, 16, 8192, 128))) fail("global B2 H16 L8192 d128", 2, 16, 8192);
    if (sched_sections_pay(2, 16, 64, 16, 1, 152, ws(2, 16, 8192, 64))) fail("global B2 H16 L8192 d64", 2, 16, 8192);
    if (sched_sections_pay(1, 2, 8, 1, 1, 152, ws(1, 2, 1024, 128))) fail("one round", 1, 2, 1024);
}

int main() {
    check_sections_choice();
    for (int lq : {1, 130, 300, 517})
        for (int lk : {1, 130, 300, 517})
            for (int wl : {-1, 0, 3, 128, 200})
                for (int wr : {-1, 0, 3, 128, 200}) check_band(lq, lk, wl, wr);
    check_dq_order();
    check_dq_semaphore_bounds({4096, 4096, 4096, 4096}, 16, false);
    check_dq_semaphore_bounds({1, 1, 1}, 3, false);
    check_dq_semaphore_bounds({300, 300}, 5, false);
    check_dq_semaphore_bounds({1, 128, 129, 0, 255, 256, 257, 1000, 1}, 4, true);
    check_dq_semaphore_bounds({127, 127, 127, 127, 127, 127, 127}, 2, true);
    check_dq_semaphore_bounds({16384, 256, 300, 4096, 1}, 16, true);
    for (int n : {1, 7, 152, 153, 1000, 1024, 4096})
        for (int grid : {1, 2, 148, 152})
            check_snake(n, grid);
    check_dense(1, 1, 1, 1);
    check_dense(2, 3, 5, 2);
    check_dense(4, 16, 16, 16);
    check_dense(2, 16, 64, 5);
    check_dense(1, 32, 128, 7);
    check_varlen({1, 128, 200, 513, 77, 256}, 3, 128, 2);
    check_varlen({1, 128, 200, 513, 77, 256}, 3, 256, 3);
    check_varlen({16384, 256, 300, 300, 4096, 1}, 16, 128, 16);
    // key lengths of their own (prefill and decode mixed; empty sides)
    for (bool over_keys : {false, true}) {
        check_varlen({1, 1, 4096, 0, 77, 513}, {8192, 300, 4096, 5, 0, 128}, 4, 128, 2, over_keys);
        check_varlen({1, 1, 4096, 0, 77, 513}, {8192, 300, 4096, 5, 0, 128}, 3, 256, 3, over_keys);
    }
    // the causal workloads of the benchmark, forward (256-row tiles) and backward (128-key blocks)
    check_causal_balance(4, 16, 4096, 256, true, 152, 0.03);
    check_causal_balance(4, 16, 4096, 128, false, 152, 0.03);
    check_causal_balance(2, 16, 8192, 256, true, 152, 0.03);
    check_causal_balance(2, 16, 8192, 128, false, 152, 0.03);
    check_causal_balance(1, 32, 32768, 256, true, 152, 0.03);
    std::printf("OK\n");
    return 0;
}
