// Backward main kernel for head dims 192 and 256.
//
// The same five MMAs, warp roles and dQ path as the d <= 128 kernel in bwd.cu
// (FlashAttention-4 paper, Section 3.2.2), with two changes forced by the
// on-chip budgets at these head dims:
//  * tensor memory (512 columns) cannot hold S^T, dP^T and full-width dK and
//    dV (2 x 128 + 2 x d > 512). A work tile is one 128-key block AND one
//    column chunk c of dK, dV and dQ: columns [128c, 128c + CW), CW = 128, or
//    64 for the second chunk at d = 192. Both chunks of a key block recompute
//    the full-d contractions S^T and dP^T (1.4x the algorithmic MMA work);
//  * shared memory (227 KB) cannot hold 128 x d tiles of K, V, Q and dO at
//    once when d = 256. K and V stay resident for the work tile; Q and dO
//    stream through a ring of 128-row x 128-column pieces, five per query
//    block in consumption order: Q[o], Q[c] (S^T), dO[o], dO[c] (dP^T; dO[c]
//    is kept for dV), then Q[c] again for dK (o = the other chunk).
// Tensor memory: S^T at 0 (P^T over it), dP^T at 128 (dS^T over it, then the
// dQ chunk), dV chunk at 256, dK chunk at 384. Every wait is bounded.
//
// A head dim of its own for v (d_qk = 192, d_v = 128, the FlashAttention-4
// paper's Section 5.1 shape): dP^T contracts over the 128 columns of V and dO,
// which are one ring piece, so a query block takes four ring items -- Q[o],
// Q[c], dO, Q[c] -- and chunk 0 owns all of dV while chunk 1 has none.
#include "kernels.h"
#include "ptx.cuh"
#include "mask.cuh"
#include "sched.cuh"
#include "dq_order.cuh"
#include "dq_reduce.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;              // query rows per Q block
constexpr int kBN = 128;              // keys per K/V block
constexpr int kThreads = 512;         // 16 warps, roles as in bwd.cu
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 16384;           // 128 rows x 64 bf16 columns
constexpr int kPieceBytes = 2 * kBox; // 128 rows x 128 columns
constexpr int kLaunchRegs = 128;
constexpr uint32_t kRegsLoadMma = 72, kRegsCompute = 128, kRegsDq = 184;
static_assert((kRegsLoadMma + 2 * kRegsCompute + kRegsDq) * 128 <= kLaunchRegs * kThreads, "register split");

__device__ __forceinline__ uint32_t packed_col(int k) { return (uint32_t)((k >> 2) * 64 + (k & 3) * 8); }

// HD: head dim of q and k; DV: of v and dO (HD, or 128 with HD = 192)
template <int HD, int DV>
struct WideBwdLayout {
    static constexpr int kHalves = HD / 64;                       // 64-column boxes per row
    static constexpr int kHalvesV = DV / 64;                      // ... of a V / dO row
    // ring items per query block: Q[o], Q[c], dO[o], dO[c], Q[c]; or Q[o], Q[c], dO, Q[c]
    static constexpr int kItems = DV == HD ? 5 : 4;
    static constexpr int kSlots = HD == 192 ? 3 : 2;                // Q/dO piece ring
    // dS tiles. The d <= 128 kernel double-buffers dS so the next dS can be
    // written while the previous dQ is staged through the other tile; here
    // shared memory has room for that only by giving up a ring slot at d = 192,
    // which measured 11% slower, so one tile.
    static constexpr int kDSTiles = 1;
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kHalves * kBox;
    static constexpr int kRingOff = kVOff + kHalvesV * kBox;
    static constexpr int kDSOff = kRingOff + kSlots * kPieceBytes;  // dS tiles, 128 x 128 bf16 (also dQ staging)
    static constexpr int kDSBytes = 2 * kBox;
    static constexpr int kStatOff = kDSOff + kDSTiles * kDSBytes;   // 2 stages: -lse2[128], -D[128]
    static constexpr int kBarOff = kStatOff + 2 * 1024;
    static constexpr int kKVFull = 0, kKVEmpty = 1, kRFull = 2, kREmpty = 2 + kSlots, kStatFull = 2 + 2 * kSlots,
                         kSFull = kStatFull + 2, kDPFull = kSFull + 1, kPFull = kDPFull + 1, kDSFull = kPFull + 1,
                         kDSEmpty = kDSFull + 1, kDQFull = kDSEmpty + 2, kDQFree = kDQFull + 1,
                         kDKVFull = kDQFree + 1, kSemGo = kDKVFull + 1,
                         kRedDone = kSemGo + 1, kDrain = kRedDone + 1,
                         kNumBars = kDrain + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16;
    static constexpr uint32_t kTS = 0, kTDP = 128, kTDV = 256, kTDK = 384;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// 64-column boxes in piece p (128-column piece p covers boxes 2p, 2p+1).
template <int HD>
__device__ __forceinline__ int piece_boxes(int p) { return min(2, HD / 64 - 2 * p); }

// Chunk width: columns of dK/dV/dQ that a work tile owns.
template <int HD>
__device__ __forceinline__ int chunk_width(int c) { return min(128, HD - 128 * c); }

struct WideBwdTile {
    int b, h, n, c;      // batch, key/value head, 128-key block, column chunk
    int lq, lk;
    int q_row0, k_row0;  // packed rows of query 0 / key 0 of the sequence
    int m_begin, m_end;  // query blocks that see this key block
    int hq0;             // first query head the tile visits
    int nblk;            // query blocks the tile visits: (group / split) x (m_end - m_begin)
    int s;               // which of the key block's split tiles (0 when split == 1)
    // block-sparse (block mask given): entry (query head h, query block m) of
    // this key block's mask column is mcol[h * mhead + m * mstride] (mhead 0:
    // one mask for all heads); nblk counts the kept pairs only
    const unsigned char* mcol;
    long mstride, mhead;
    int nheads;          // query heads the tile visits
};

// The tile's query blocks in visiting order: every query head of the tile's
// share of the group, each over [m_begin, m_end).
struct WideQWalk {
    int h, m;   // query head, 128-row query block
    template <bool kGQA>
    __device__ __forceinline__ void next(const WideBwdTile& f) {
        ++m;
        if (kGQA && m == f.m_end) {
            m = f.m_begin;
            ++h;
        }
    }
};
__device__ __forceinline__ WideQWalk qwalk(const WideBwdTile& f) { return WideQWalk{f.hq0, f.m_begin}; }

// Block-sparse walk: from (qw.h, qw.m) on, the first pair the block mask keeps
// (warp-wide scans: every lane of the warp calls it alike).
__device__ __forceinline__ void sparse_seek(const WideBwdTile& f, WideQWalk& qw, int lane) {
    while (qw.h < f.hq0 + f.nheads) {
        qw.m = sparse_next_col(f.mcol + qw.h * f.mhead, f.mstride, qw.m, f.m_end, lane);
        if (qw.m < f.m_end) return;
        ++qw.h;
        qw.m = f.m_begin;
    }
}

// The first pair of the tile's walk, and the next one.
template <bool kSparse>
__device__ __forceinline__ WideQWalk qwalk_start(const WideBwdTile& f, int lane) {
    WideQWalk qw = qwalk(f);
    if (kSparse && f.mcol) sparse_seek(f, qw, lane);
    return qw;
}
template <bool kGQA, bool kSparse>
__device__ __forceinline__ void qwalk_step(WideQWalk& qw, const WideBwdTile& f, int lane) {
    if (kSparse && f.mcol) {
        ++qw.m;
        sparse_seek(f, qw, lane);
    } else {
        qw.next<kGQA>(f);
    }
}


// Tile t: key-block tile t/2 of the d <= 128 walk (split tiles included), chunk
// t%2 (the two chunks of a key block run at the same time on neighbouring CTAs
// and share its loads in L2).
// kGQA: grouped heads, as in bwd.cu's bwd_tile
__device__ __forceinline__ int floor_div_w(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// kBand, kSparse: as in bwd.cu's bwd_tile
// kSpt (the deterministic kernels): with a right mask bound, key blocks are
// walked shortest first -- the last key block of a (batch, head) first -- so
// that, with each dQ tile's contributions serialised from its highest key
// block down, no work tile waits at its first dQ write (FlashAttention-4
// paper, Section 3.2.4, SPT order).
template <bool kGQA, bool kBand, bool kSparse, bool kSpt>
__device__ __forceinline__ WideBwdTile wide_bwd_tile(int t, const BwdParams& p, const VarlenMap* vm, int lane) {
    const Geometry& g = p.g;
    const int sp = kGQA ? (t >> 1) % p.split : 0;
    const int u = kGQA ? (t >> 1) / p.split : t >> 1;
    const bool spt = kSpt && g.causal;
    Tile ti = vm ? sched_varlen(*vm, u, g.B, g.Hkv, kBN, p.head_section, spt, true)
                 : (g.causal ? sched_dense_lpt(u, g.B, g.Hkv, p.nm, spt)
                             : sched_dense(u, g.Hkv, p.nm, p.head_section, false));
    WideBwdTile f;
    f.b = ti.b;
    f.h = ti.h;
    f.n = ti.m;
    f.c = t & 1;
    if (vm) {
        f.lq = vm_lq(*vm, ti.b);
        f.lk = vm_lk(*vm, ti.b);
        f.q_row0 = vm->start[ti.b];
        f.k_row0 = vm->start_k[ti.b];
    } else {
        f.lq = g.Lq;
        f.lk = g.Lk;
        f.q_row0 = ti.b * g.Lq;
        f.k_row0 = ti.b * g.Lk;
    }
    // the query blocks whose rows see some key of this block (the mask band;
    // none: the tile writes zero dK/dV rows). No mask or the causal one: all
    // blocks, or those from the one holding row n*kBN - (lk - lq) on.
    if constexpr (kBand) {
        band_query_blocks(mask_band(f.lq, f.lk, g.win_left, g.win_right), f.n * kBN, f.n * kBN + kBN - 1, kBM,
                          &f.m_begin, &f.m_end);
    } else {
        f.m_end = (f.lq + kBM - 1) / kBM;
        f.m_begin = 0;
        if (g.causal) f.m_begin = max(0, floor_div_w(f.n * kBN - (f.lk - f.lq), kBM));
        if (f.n * kBN >= f.lk) f.m_end = f.m_begin;
    }
    if constexpr (kGQA) {
        const int per = g.group / p.split;
        f.s = sp;
        f.hq0 = f.h * g.group + sp * per;
        f.nblk = per * (f.m_end - f.m_begin);
    } else {
        f.s = 0;
        f.hq0 = f.h;
        f.nblk = f.m_end - f.m_begin;
    }
    f.mcol = nullptr;
    if constexpr (kSparse) {
        f.mstride = f.mhead = 0;
        f.nheads = f.m_end > f.m_begin ? f.nblk / (f.m_end - f.m_begin) : 0;
        if (p.mask.ptr) {   // keep the (head, query block) pairs the block mask keeps
            f.mcol = p.mask.ptr + f.n;
            f.mstride = mask_cols(g);
            f.mhead = p.mask.heads == 1 ? 0 : (long)mask_rows(g) * mask_cols(g);
            int kept = 0;
            if (f.nheads > 0) {
                if (f.mhead == 0) {
                    kept = f.nheads * sparse_count_col(f.mcol, f.mstride, f.m_begin, f.m_end, lane);
                } else {
                    for (int x = 0; x < f.nheads; ++x)
                        kept += sparse_count_col(f.mcol + (f.hq0 + x) * f.mhead, f.mstride, f.m_begin, f.m_end, lane);
                }
            }
            f.nblk = kept;
        }
    }
    return f;
}

// kDet: deterministic dQ accumulation (a separate instantiation keeps the
// other path's code out of each kernel); kGQA: grouped heads; kBand: the mask
// has a left bound (as in bwd.cu)
template <int HD, int DV, bool kDet, bool kGQA, bool kBand, bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
bwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                const __grid_constant__ CUtensorMap tmDQ, const BwdParams p, const VarlenMap* vm) {
    using Lay = WideBwdLayout<HD, DV>;
    constexpr int NS = Lay::kSlots;
    constexpr int kItemsPerBlock = Lay::kItems;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Geometry& g = p.g;
    if (base & 1023u) {
        if (tid == 0) atomicCAS(p.status, kStatusOk, kStatusMisaligned);
        return;
    }
    auto bar = [&](int i) -> uint32_t { return base + Lay::kBarOff + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kMiscOff + 4);

    if (tid == 0) {
        mbar_init(bar(Lay::kKVFull), 1);
        mbar_init(bar(Lay::kKVEmpty), 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(Lay::kRFull + s), 1);
            mbar_init(bar(Lay::kREmpty + s), 1);
        }
        mbar_init(bar(Lay::kStatFull + 0), 1);
        mbar_init(bar(Lay::kStatFull + 1), 1);
        mbar_init(bar(Lay::kSFull), 1);
        mbar_init(bar(Lay::kDPFull), 1);
        mbar_init(bar(Lay::kPFull), 256);
        mbar_init(bar(Lay::kDSFull), 256);
        mbar_init(bar(Lay::kDSEmpty + 0), 4);   // each dQ warp releases its rows of the stage
        mbar_init(bar(Lay::kDSEmpty + 1), 4);
        mbar_init(bar(Lay::kDQFull), 1);
        mbar_init(bar(Lay::kDQFree), 128);
        mbar_init(bar(Lay::kDKVFull), 1);
        mbar_init(bar(Lay::kSemGo), 1);
        mbar_init(bar(Lay::kRedDone), 4);       // deterministic: each dQ warp's adds are complete
        mbar_init(bar(Lay::kDrain), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmDO);
        tma_prefetch_desc(&tmDQ);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{abort_flag, p.status, p.wait_budget_ns};
    const bool varlen = g.cu_seqlens != nullptr;
    const VarlenMap* vmp = varlen ? vm : nullptr;
    const int n_tiles = 2 * (varlen ? vm->pre[g.B] * (kGQA ? p.split : 1) : p.n_tiles);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        setmaxnreg_dec<kRegsLoadMma>();
        uint32_t tile_it = 0, ic = 0, qb = 0;
        bool ok = true;
        float* stats = reinterpret_cast<float*>(smem + Lay::kStatOff);
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const WideBwdTile f = wide_bwd_tile<kGQA, kBand, kSparse, kDet>(t, p, vmp, lane);
            if (kSparse ? f.nblk == 0 : f.m_begin >= f.m_end) continue;
            ok = warp_wait(bar(Lay::kKVEmpty), (tile_it & 1u) ^ 1u, w, lane);
            if (!ok) break;
            if (lane == 0) {
                mbar_expect_tx(bar(Lay::kKVFull), (Lay::kHalves + Lay::kHalvesV) * kBox);
                for (int hf = 0; hf < Lay::kHalves; ++hf)
                    tma_load_3d(base + Lay::kKOff + hf * kBox, &tmK, bar(Lay::kKVFull), hf * 64, f.h,
                                f.k_row0 + f.n * kBN);
                for (int hf = 0; hf < Lay::kHalvesV; ++hf)
                    tma_load_3d(base + Lay::kVOff + hf * kBox, &tmV, bar(Lay::kKVFull), hf * 64, f.h,
                                f.k_row0 + f.n * kBN);
            }
            __syncwarp();
            ++tile_it;
            const int pc = f.c, po = 1 - f.c;
            WideQWalk qw = qwalk_start<kSparse>(f, lane);
            for (int u = 0; u < f.nblk && ok; ++u, qwalk_step<kGQA, kSparse>(qw, f, lane)) {
                const int m = qw.m;
                for (int item = 0; item < kItemsPerBlock; ++item) {
                    const uint32_t slot = ic % NS;
                    ok = warp_wait(bar(Lay::kREmpty + slot), ((ic / NS) & 1u) ^ 1u, w, lane);
                    if (!ok) break;
                    if (item == 0) {
                        // row statistics of this query block, negated (-lse in log2 units, -D); the
                        // stage is free: its previous block's dS was consumed before the
                        // ring slot just acquired could be released
                        float* nlse2 = stats + (qb & 1u) * 256;
                        float* ndd = nlse2 + 128;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int r = m * kBM + lane * 4 + e;
                            float lv = -INFINITY, dv = 0.f;   // negated; rows past the end: P = 0
                            if (r < f.lq) {
                                const long si = varlen ? (long)qw.h * g.Lq + f.q_row0 + r
                                                       : ((long)f.b * g.H + qw.h) * g.Lq + r;
                                lv = -p.lse[si] * kLog2e;
                                dv = -p.delta[si];
                            }
                            nlse2[lane * 4 + e] = lv;
                            ndd[lane * 4 + e] = dv;
                        }
                        __threadfence_block();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(Lay::kStatFull + (qb & 1u)));
                    }
                    int piece, nb;
                    const CUtensorMap* src;
                    if constexpr (Lay::kItems == 5) {
                        piece = (item == 0 || item == 2) ? po : pc;
                        nb = piece_boxes<HD>(piece);
                        src = (item == 2 || item == 3) ? &tmDO : &tmQ;
                    } else {   // item 2: the whole of dO (one piece)
                        piece = item == 0 ? po : (item == 2 ? 0 : pc);
                        nb = item == 2 ? Lay::kHalvesV : piece_boxes<HD>(piece);
                        src = item == 2 ? &tmDO : &tmQ;
                    }
                    if (lane == 0) {
                        mbar_expect_tx(bar(Lay::kRFull + slot), nb * kBox);
                        for (int bb = 0; bb < nb; ++bb)
                            tma_load_3d(base + Lay::kRingOff + slot * kPieceBytes + bb * kBox, src,
                                        bar(Lay::kRFull + slot), (2 * piece + bb) * 64, qw.h, f.q_row0 + m * kBM);
                    }
                    __syncwarp();
                    ++ic;
                }
                ++qb;
            }
        }
        if (lane == 0) {
            if (tile_it) drain_wait(bar(Lay::kKVFull), (tile_it - 1) & 1u, p.wait_budget_ns);
            for (uint32_t i = 0; i < (uint32_t)NS && i < ic; ++i) {
                const uint32_t n = ic - 1 - i;
                drain_wait(bar(Lay::kRFull + n % NS), (n / NS) & 1u, p.wait_budget_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        setmaxnreg_dec<kRegsLoadMma>();
        constexpr uint32_t kIdSq = idesc_bf16_f32(kBN, kBM, false, false);
        constexpr uint32_t kIdKV128 = idesc_bf16_f32(kBN, 128, false, true);
        constexpr uint32_t kIdKV64 = idesc_bf16_f32(kBN, 64, false, true);
        constexpr uint32_t kIdDQ128 = idesc_bf16_f32(kBM, 128, true, true);
        constexpr uint32_t kIdDQ64 = idesc_bf16_f32(kBM, 64, true, true);
        const SmemDesc k_km = sdesc_sw128_split(base + Lay::kKOff, 16, 1024);
        const SmemDesc v_km = sdesc_sw128_split(base + Lay::kVOff, 16, 1024);
        const SmemDesc k_mn = sdesc_sw128_split(base + Lay::kKOff, kBox, 1024);
        const SmemDesc ds_mn0 = sdesc_sw128_split(base + Lay::kDSOff, kBox, 1024);
        const SmemDesc r_km0 = sdesc_sw128_split(base + Lay::kRingOff, 16, 1024);
        const SmemDesc r_mn0 = sdesc_sw128_split(base + Lay::kRingOff, kBox, 1024);
        auto at_slot = [&](SmemDesc d, uint32_t slot) {
            d.lo += slot * desc_step(kPieceBytes);
            return d;
        };
        // wait for ring item `item` (global index) to land; returns its slot
        auto item_wait = [&](uint32_t item, uint32_t& slot) -> bool {
            slot = item % NS;
            return warp_wait(bar(Lay::kRFull + slot), (item / NS) & 1u, w, lane);
        };
        // D[128 x 128] (+)= A[128 x 128c'] B^T over one piece: A = K or V boxes
        // 2*piece.., B = the piece in ring slot `slot`; both K-major
        auto mma_piece = [&](uint32_t d_tmem, SmemDesc a, int piece, uint32_t slot, bool acc) {
            const SmemDesc b = at_slot(r_km0, slot);
            const int nb = piece_boxes<HD>(piece);
            for (int bb = 0; bb < nb; ++bb) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t a_off = desc_step((2 * piece + bb) * kBox + k * 32);
                    const uint32_t b_off = desc_step(bb * kBox + k * 32);
                    mma_ss(d_tmem, a, a_off, b, b_off, kIdSq, (acc || bb > 0 || k > 0) ? 1u : 0u);
                }
            }
        };
        uint32_t tile_it = 0, qb = 0, pcnt = 0, dsc = 0, dqf = 0;
        bool ok = true;
        // S^T of query block `blk` (its items 0 and 1)
        auto issue_s = [&](uint32_t blk, int pc, int po) -> bool {
            const uint32_t i0 = blk * kItemsPerBlock;
            uint32_t s0, s1;
            if (!item_wait(i0, s0) || !item_wait(i0 + 1, s1)) return false;
            tc_fence_after_sync();
            if (lane == 0) {
                mma_piece(tmem + Lay::kTS, k_km, po, s0, false);
                mma_piece(tmem + Lay::kTS, k_km, pc, s1, true);
                tc_commit(bar(Lay::kSFull));
                tc_commit(bar(Lay::kREmpty + s0));
                tc_commit(bar(Lay::kREmpty + s1));
            }
            __syncwarp();
            return true;
        };
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const WideBwdTile f = wide_bwd_tile<kGQA, kBand, kSparse, kDet>(t, p, vmp, lane);
            if (kSparse ? f.nblk == 0 : f.m_begin >= f.m_end) continue;
            const int pc = f.c, po = 1 - f.c;
            const bool narrow = chunk_width<HD>(f.c) == 64;
            const uint32_t id_kv = narrow ? kIdKV64 : kIdKV128;
            const uint32_t id_dq = narrow ? kIdDQ64 : kIdDQ128;
            const SmemDesc kc_mn = [&] {   // K columns of this chunk, MN-major (B of dQ)
                SmemDesc d = k_mn;
                d.lo += desc_step(2 * f.c * kBox);
                return d;
            }();
            ok = warp_wait(bar(Lay::kKVFull), tile_it & 1u, w, lane);
            if (!ok) break;
            ++tile_it;
            tc_fence_after_sync();
            ok = issue_s(qb, pc, po);
            if (!ok) break;
            for (int u = 0; u < f.nblk; ++u) {
                const uint32_t i0 = qb * kItemsPerBlock;
                const bool more = u + 1 < f.nblk;
                // dP^T = V dO^T once the previous dQ chunk has left tensor memory
                ok = warp_wait(bar(Lay::kDQFree), (dqf & 1u) ^ 1u, w, lane);
                if (!ok) break;
                ++dqf;
                uint32_t s2, s3 = 0, s4;
                ok = item_wait(i0 + 2, s2) && (Lay::kItems == 4 || item_wait(i0 + 3, s3));
                if (!ok) break;
                tc_fence_after_sync();
                if (lane == 0) {
                    if constexpr (Lay::kItems == 5) {
                        mma_piece(tmem + Lay::kTDP, v_km, po, s2, false);
                        mma_piece(tmem + Lay::kTDP, v_km, pc, s3, true);
                        tc_commit(bar(Lay::kREmpty + s2));
                    } else {   // over the DV columns of V and of the one dO piece
                        const SmemDesc b = at_slot(r_km0, s2);
#pragma unroll
                        for (int bb = 0; bb < Lay::kHalvesV; ++bb)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint32_t off = desc_step(bb * kBox + kk * 32);
                                mma_ss(tmem + Lay::kTDP, v_km, off, b, off, kIdSq, (bb > 0 || kk > 0) ? 1u : 0u);
                            }
                    }
                    tc_commit(bar(Lay::kDPFull));
                }
                __syncwarp();
                // dV[:, chunk] += P^T dO[:, chunk] (P^T from tensor memory); with DV < HD
                // chunk 0 owns all of dV and chunk 1 none
                ok = warp_wait(bar(Lay::kPFull), pcnt & 1u, w, lane);
                if (!ok) break;
                ++pcnt;
                tc_fence_after_sync();
                if (lane == 0) {
                    const uint32_t s_do = Lay::kItems == 5 ? s3 : s2;
                    if (Lay::kItems == 5 || f.c == 0) {
                        const SmemDesc do_mn = at_slot(r_mn0, s_do);
#pragma unroll
                        for (int kk = 0; kk < kBM / 16; ++kk)
                            mma_ts(tmem + Lay::kTDV, tmem + Lay::kTS + packed_col(kk), do_mn, desc_step(kk * 2048),
                                   id_kv, (u > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(bar(Lay::kREmpty + s_do));
                }
                __syncwarp();
                // dK[:, chunk] += dS^T Q[:, chunk]; dQ[:, chunk] = dS K[:, chunk]
                ok = warp_wait(bar(Lay::kDSFull), dsc & 1u, w, lane);
                if (!ok) break;
                ++dsc;
                ok = item_wait(i0 + kItemsPerBlock - 1, s4);
                if (!ok) break;
                tc_fence_after_sync();
                if (lane == 0) {
                    const SmemDesc q_mn = at_slot(r_mn0, s4);
                    SmemDesc ds_mn = ds_mn0;   // this block's dS tile
                    ds_mn.lo += (qb % Lay::kDSTiles) * desc_step(Lay::kDSBytes);
#pragma unroll
                    for (int kk = 0; kk < kBM / 16; ++kk)
                        mma_ts(tmem + Lay::kTDK, tmem + Lay::kTDP + packed_col(kk), q_mn, desc_step(kk * 2048), id_kv,
                               (u > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        mma_ss(tmem + Lay::kTDP, ds_mn, desc_step(kk * 2048), kc_mn, desc_step(kk * 2048), id_dq,
                               kk > 0 ? 1u : 0u);
                    tc_commit(bar(Lay::kDQFull));
                    tc_commit(bar(Lay::kREmpty + s4));
                    if (!more) {
                        tc_commit(bar(Lay::kDKVFull));
                        tc_commit(bar(Lay::kKVEmpty));
                    }
                }
                __syncwarp();
                ++qb;
                // the next S^T only now: issued before dK/dQ it delayed the dQ read-out
                // and the next dP^T behind it (measured 22% slower at d = 192)
                if (more) {
                    ok = issue_s(qb, pc, po);
                    if (!ok) break;
                }
            }
        }
        if (lane == 0) {
            tc_commit(bar(Lay::kDrain));
            drain_wait(bar(Lay::kDrain), 0, p.wait_budget_ns);
        }
        __syncwarp();
    } else if (warp < 4) {
        setmaxnreg_dec<kRegsLoadMma>();
    } else if (warp < 12) {
        // ------------------------------------------------------------ compute warpgroups
        const int wg = (warp - 4) >> 2;            // query columns [64*wg, 64*wg + 64)
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;         // key row inside the block
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = g.scale_log2;
        uint8_t* const ds_tiles = smem + Lay::kDSOff + wg * kBox;
        const float* stats = reinterpret_cast<const float*>(smem + Lay::kStatOff);
        uint32_t sc = 0, qb = 0, dpc = 0, dsw = 0, tile_it = 0;
        bool ok = true;
        uint32_t rr[32];
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const WideBwdTile f = wide_bwd_tile<kGQA, kBand, kSparse, kDet>(t, p, vmp, lane);
            const int cw = chunk_width<HD>(f.c);
            const int key = f.n * kBN + r;
            const bool key_ok = key < f.lk;
            const long krow = (long)f.k_row0 + key;
            // this thread's dK/dV chunk row: bf16 outputs, or (split tiles) fp32
            // partial slots, dK slot f.s and dV slot split + f.s; computed where
            // used, so that no pointer stays live through the query-block loop
            const bool partial = kGQA && p.split > 1;
            // columns of the chunk: cw of dK; of dV cw too, or with DV < HD all DV
            // columns in chunk 0 and none in chunk 1
            const int cwv = DV == HD ? cw : (f.c == 0 ? DV : 0);
            auto kv_off = [&](int which) {   // 0: dV (rows of DV), 1: dK (rows of HD)
                return which ? (krow * g.Hkv + f.h) * HD + 128 * f.c + wg * (cw / 2)
                             : (krow * g.Hkv + f.h) * DV + 128 * f.c + wg * (cwv / 2);
            };
            auto part_slot = [&](int which) {   // dK slots (HD wide) first, then the dV slots (DV wide)
                const long rows = (varlen ? (long)g.Lk : (long)g.B * g.Lk) * g.Hkv;
                return p.dkv_part + (which ? f.s * rows * HD : (p.split * HD + f.s * DV) * rows) + kv_off(which);
            };
            if (kSparse ? f.nblk == 0 : f.m_begin >= f.m_end) {   // no query sees this key block
                if (key_ok) {
                    for (int which = 0; which < 2; ++which) {
                        const int cols = (which ? cw : cwv) / 2;
                        if (partial) {
                            float4* z = reinterpret_cast<float4*>(part_slot(which));
                            for (int c = 0; c < cols / 4; ++c) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                        } else {
                            uint4* z = reinterpret_cast<uint4*>((which ? p.dk : p.dv) + kv_off(which));
                            for (int c = 0; c < cols / 8; ++c) z[c] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                continue;
            }
            // query q is allowed for this key iff q_lo <= q < q_hi (the mask band)
            int q_lo, q_hi;
            if constexpr (kBand) {
                const MaskBand mb = mask_band(f.lq, f.lk, g.win_left, g.win_right);
                q_lo = key_ok ? band_query_lo(mb, key) : 0;
                q_hi = key_ok ? band_query_hi(mb, key) : 0;   // (key_ok false: lo = 64 below)
            } else {
                q_lo = g.causal ? key - (f.lk - f.lq) : 0;
                q_hi = f.lq;
            }
            WideQWalk qw = qwalk_start<kSparse>(f, lane);
            for (int u = 0; u < f.nblk; ++u, qwalk_step<kGQA, kSparse>(qw, f, lane)) {
                const int m = qw.m;
                ok = warp_wait(bar(Lay::kSFull), sc & 1u, w, lane);
                if (!ok) break;
                ++sc;
                ok = warp_wait(bar(Lay::kStatFull + (qb & 1u)), (qb >> 1) & 1u, w, lane);
                if (!ok) break;
                const uint32_t stage = qb & 1u;
                ++qb;
                tc_fence_after_sync();
                float pv[64];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    tmem_ld32(tmem + lane_off + Lay::kTS + wg * 64 + c * 32, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) pv[c * 32 + i] = u2f(rr[i]);
                }
                // the producer stages -lse (log2 units) and -D, so both steps are packed fp32 pairs
                const float* nlse2 = stats + stage * 256 + wg * 64;
                const float* ndd = stats + stage * 256 + 128 + wg * 64;
                const int q0 = m * kBM + wg * 64;
                const bool full = key_ok && q0 >= q_lo && q0 + 64 <= q_hi;
                const uint64_t sc2 = f32x2(sl2, sl2);
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const float2 nl = *reinterpret_cast<const float2*>(nlse2 + c);
                    float x0, x1;
                    f32x2_split(ffma2(f32x2(pv[c], pv[c + 1]), sc2, f32x2(nl.x, nl.y)), x0, x1);
                    pv[c] = ex2_mufu(x0);
                    pv[c + 1] = ex2_mufu(x1);
                }
                if (!full) {   // diagonal or ragged block: keep query columns [lo, hi) only
                    const int lo = key_ok ? q_lo - q0 : 64, hi = q_hi - q0;
#pragma unroll
                    for (int c = 0; c < 64; ++c) pv[c] = (c >= lo && c < hi) ? pv[c] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) rr[i] = pack_bf16x2(pv[2 * i], pv[2 * i + 1]);
                tmem_st32(tmem + lane_off + Lay::kTS + wg * 64, rr);
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(bar(Lay::kPFull));
                // dS^T = P^T * (dP^T - D)
                ok = warp_wait(bar(Lay::kDPFull), dpc & 1u, w, lane);
                if (!ok) break;
                ++dpc;
                tc_fence_after_sync();
                const uint32_t dsb = dsw % Lay::kDSTiles;   // alternate dS tiles per block (d = 192)
                uint8_t* ds_tile = ds_tiles + dsb * Lay::kDSBytes;
                ok = warp_wait(bar(Lay::kDSEmpty + dsb), ((dsw / Lay::kDSTiles) & 1u) ^ 1u, w, lane);
                if (!ok) break;
                ++dsw;
                uint32_t ds2[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    tmem_ld32(tmem + lane_off + Lay::kTDP + wg * 64 + c * 32, rr);
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int cc = c * 32 + i + 2 * e;
                            const float2 nd = *reinterpret_cast<const float2*>(ndd + cc);
                            float d0, d1;
                            f32x2_split(fmul2(f32x2(pv[cc], pv[cc + 1]),
                                              fadd2(f32x2(u2f(rr[i + 2 * e]), u2f(rr[i + 2 * e + 1])), f32x2(nd.x, nd.y))),
                                        d0, d1);
                            ds2[cc >> 1] = pack_bf16x2(d0, d1);
                        }
                        // 128-byte swizzle: 16-byte chunk j of row r lands at chunk j ^ (r % 8)
                        const int chunk = (c * 32 + i) >> 3;
                        uint8_t* dst = ds_tile + (r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4);
                        const int b = (c * 32 + i) >> 1;
                        *reinterpret_cast<uint4*>(dst) = make_uint4(ds2[b], ds2[b + 1], ds2[b + 2], ds2[b + 3]);
                    }
                }
                tmem_st32(tmem + lane_off + Lay::kTDP + wg * 64, ds2);
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(bar(Lay::kDSFull));
            }
            if (!ok) break;
            // epilogue: cw/2 columns of the dV and dK chunks for this key row
            ok = warp_wait(bar(Lay::kDKVFull), tile_it & 1u, w, lane);
            if (!ok) break;
            ++tile_it;
            tc_fence_after_sync();
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const int cols = which ? cw : cwv;
                const uint32_t tcol = (which ? Lay::kTDK : Lay::kTDV) + wg * (cols / 2);
                const float mul = which ? g.scale : 1.f;
                __nv_bfloat16* dst = (which ? p.dk : p.dv) + kv_off(which);
                float* pdst = partial ? part_slot(which) : nullptr;
                for (int c = 0; c < cols / 64; ++c) {
                    tmem_ld32(tmem + lane_off + tcol + c * 32, rr);
                    if (key_ok && partial) {   // unscaled: the sum kernel scales dK
                        float4* d4 = reinterpret_cast<float4*>(pdst + c * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4)
                            d4[v4] = make_float4(u2f(rr[4 * v4]), u2f(rr[4 * v4 + 1]), u2f(rr[4 * v4 + 2]),
                                                 u2f(rr[4 * v4 + 3]));
                    } else if (key_ok) {
                        uint32_t o2[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) o2[i] = pack_bf16x2(u2f(rr[2 * i]) * mul, u2f(rr[2 * i + 1]) * mul);
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            d4[v4] = make_uint4(o2[4 * v4], o2[4 * v4 + 1], o2[4 * v4 + 2], o2[4 * v4 + 3]);
                    }
                }
            }
            tc_fence_before_sync();
        }
    } else {
        // ------------------------------------------------------------ dQ read-out warpgroup
        // As in bwd.cu, for one column chunk: each warp adds its own 32 rows with
        // TMA reduce-adds staged through this block's dS tile (dq_reduce.cuh);
        // deterministic mode: the same reduce-adds under the chunk's semaphore,
        // every warp's completing before the next key block's start.
        const int quarter = warp & 3;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        setmaxnreg_inc<kRegsDq>();
        const bool leader = warp == 12 && lane == 0;
        uint32_t dqc = 0, sgo = 0, rdc = 0;
        bool ok = true;
        uint32_t rr[32];
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const WideBwdTile f = wide_bwd_tile<kGQA, kBand, kSparse, kDet>(t, p, vmp, lane);
            const int cw = chunk_width<HD>(f.c);
            const int rounds = cw / 64;
            WideQWalk qw = qwalk_start<kSparse>(f, lane);
            for (int u = 0; u < f.nblk; ++u, qwalk_step<kGQA, kSparse>(qw, f, lane)) {
                const int m = qw.m;
                ok = warp_wait(bar(Lay::kDQFull), dqc & 1u, w, lane);
                if (!ok) break;
                const uint32_t dsb = dqc % Lay::kDSTiles;   // the dS tile this block's dQ MMA read
                uint8_t* stage = smem + Lay::kDSOff + dsb * Lay::kDSBytes;
                const uint32_t stage_s = base + Lay::kDSOff + dsb * Lay::kDSBytes;
                ++dqc;
                tc_fence_after_sync();
                int* sem = nullptr;
                if constexpr (kDet) {
                    // this block's turn at chunk c of the dQ tile (the order of bwd.cu, one
                    // semaphore per chunk): the leader waits for it and tells the warpgroup
                    sem = p.semaphores + 2 * dq_semaphore(p, f, qw.h, m, varlen) + f.c;
                    if (leader) {
                        if (sem_wait(sem, dq_turn<kBand, kSparse>(p, f, qw.h, m), w)) fence_proxy_async_global();
                        mbar_arrive(bar(Lay::kSemGo));
                    }
                    ok = warp_wait(bar(Lay::kSemGo), sgo & 1u, w, lane);
                    ++sgo;
                    ok = ok && !*abort_flag;
                    if (!ok) break;
                }
                uint32_t row[128];
                if (rounds == 2) {
                    tmem_ld128(tmem + lane_off + Lay::kTDP, row);
                } else {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        tmem_ld32(tmem + lane_off + Lay::kTDP + c * 32, rr);
#pragma unroll
                        for (int i = 0; i < 32; ++i) row[c * 32 + i] = rr[i];
                    }
                }
                tc_fence_before_sync();
                mbar_arrive(bar(Lay::kDQFree));
                dq_warp_reduce(&tmDQ, stage, stage_s, row, rounds, 128 * f.c, qw.h, f.q_row0 + m * kBM, quarter,
                               lane);
                if (lane == 0) {
                    if constexpr (kDet) {
                        bulk_wait_group0();   // this warp's adds are complete
                        fence_proxy_async_global();
                        mbar_arrive(bar(Lay::kRedDone));
                    } else {
                        bulk_wait_group_read0();
                    }
                    mbar_arrive(bar(Lay::kDSEmpty + dsb));   // this warp's rows of the stage are read
                }
                if constexpr (kDet) {
                    if (leader && mbar_wait(bar(Lay::kRedDone), rdc & 1u, w))
                        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sem) : "memory");
                    ++rdc;
                }
                __syncwarp();
            }
        }
        if (lane == 0) bulk_wait_group0();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// The instantiation for a mask: none or causal; a general band; a band with a block mask.
template <int HD, int DV, bool kDet, bool kGQA>
auto wide_kernel_for(bool band, bool sparse) {
    return sparse ? bwd_wide_kernel<HD, DV, kDet, kGQA, true, true>
                  : (band ? bwd_wide_kernel<HD, DV, kDet, kGQA, true, false>
                          : bwd_wide_kernel<HD, DV, kDet, kGQA, false, false>);
}

template <int HD, int DV>
cudaError_t launch_wide_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p, const VarlenMap* vm,
                           int num_sms, cudaStream_t stream) {
    using Lay = WideBwdLayout<HD, DV>;
    const bool gqa = p.g.group > 1, sparse = p.mask.ptr != nullptr;
    const bool band = sparse || p.g.win_left >= 0 || p.g.win_right > 0;
    auto kern = p.deterministic ? (gqa ? wide_kernel_for<HD, DV, true, true>(band, sparse)
                                       : wide_kernel_for<HD, DV, true, false>(band, sparse))
                                : (gqa ? wide_kernel_for<HD, DV, false, true>(band, sparse)
                                       : wide_kernel_for<HD, DV, false, false>(band, sparse));
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    const int grid = p.g.cu_seqlens ? num_sms : min(2 * p.n_tiles, num_sms);
    if (grid <= 0) return cudaSuccess;
    kern<<<grid, kThreads, Lay::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, p, vm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                            const void* varlen_map, int num_sms, cudaStream_t stream) {
    const VarlenMap* vm = static_cast<const VarlenMap*>(varlen_map);
    if (p.g.d == 192 && p.d_v == 128) return launch_wide_hd<192, 128>(tq, tk, tv, tdo, tdq, p, vm, num_sms, stream);
    if (p.d_v != p.g.d) return cudaErrorInvalidValue;
    switch (p.g.d) {
        case 192: return launch_wide_hd<192, 192>(tq, tk, tv, tdo, tdq, p, vm, num_sms, stream);
        case 256: return launch_wide_hd<256, 256>(tq, tk, tv, tdo, tdq, p, vm, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
