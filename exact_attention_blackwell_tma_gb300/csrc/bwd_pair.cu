// Backward pass on CTA pairs: the main kernel of dQ, dK, dV with 2-CTA tensor
// cores (tcgen05 .cta_group::2), head dims 64 and 128.
//
// FlashAttention-4 paper, Section 3.2.3 "2-CTA backward pass": with M = 256
// the two CTAs of a cluster act as one larger tile -- each stages half of
// operand B in its own shared memory and keeps its own slice of the
// accumulator -- which cuts the shared-memory operand traffic that bounds the
// backward; the pair also restructures the dQ accumulation so that half as
// many global reduce-adds are issued (Section 7). Section 2.2: one thread of
// the pair issues each MMA, the peer CTA must stay resident while it runs, and
// a kernel that uses the pair mode uses it for every tensor-memory and
// tensor-core instruction.
//
// Work tile: one key-block pair (256 keys) of one (batch, key/value head); CTA
// r of the cluster owns key block 2p + r. Both walk the query blocks either key
// block sees, for every query head of the key/value head's group (grouped
// heads), in the same order; dK and dV sum over the group in the tile. Per query block (128 queries) the even CTA's MMA
// thread issues:
//   S^T  = K Q^T     M = 256 (keys), N = 128 (queries); B = Q split by query halves
//   dP^T = V dO^T    M = 256, N = 128;                  B = dO split by query halves
//   dV  += P^T dO    M = 256, N = d;  A = P^T from each CTA's tensor memory,
//                                     B = dO split by column halves
//   dK  += dS^T Q    M = 256, N = d;  A = dS^T from tensor memory, B = Q split
//                                     by column halves
//   dQ   = dS K      M = 128 (queries: 64 per CTA), N = d, K = the pair's 256
//                    keys; A = dS of this CTA's 64 queries over both key blocks (the
//                    peer writes its half into this CTA's shared memory), B = K of the
//                    256 keys, this CTA's d/2 columns
// so each CTA adds a 64 x d dQ tile per query block to the fp32 accumulator:
// per pair one reduce-add pass per 256 keys instead of two.
//
// The column halves of B (the MN-major operands of dV, dK, dQ) are 64 columns
// with the 128-byte swizzle at d = 128 and 32 columns (64 bytes a row) with the
// 64-byte swizzle at d = 64; everything else is the same at both head dims.
//
// Roles per CTA (512 threads): warp 0 loads (TMA; the pair's loads of one MMA
// complete on the even CTA's barrier), warp 1 issues the MMAs (even CTA only),
// warps 4-11 two compute warpgroups (query columns 0-63 / 64-127, one key row
// per thread), warps 12-15 the dQ warpgroup (read-out, staging through the
// finished Q stage, TMA reduce-adds). Every wait is bounded; on a timeout the
// CTA stops issuing work, drains what it issued, frees tensor memory and
// returns, and its peer times out in turn.
#include "kernels.h"
#include "ptx.cuh"
#include "mask.cuh"
#include "sched.cuh"
#include "dq_order.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;              // query rows per query block
constexpr int kBN = 128;              // keys per key block (one CTA)
constexpr int kThreads = 512;
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 16384;           // 128 rows x 64 bf16 columns
constexpr int kQuad = 8192;           // 64 rows x 64 bf16 columns
constexpr int kLaunchRegs = 128;
constexpr uint32_t kRegsLoadMma = 72, kRegsCompute = 128, kRegsDq = 184;
static_assert((kRegsLoadMma + 2 * kRegsCompute + kRegsDq) * 128 <= kLaunchRegs * kThreads, "register split");

__device__ __forceinline__ uint32_t packed_col(int k) { return (uint32_t)((k >> 2) * 64 + (k & 3) * 8); }

template <int HD>
struct PairLay {
    static constexpr bool kNarrow = HD == 64;   // column halves of 32: the 64-byte swizzle
    static constexpr int kQStages = 2;
    // A Q (dO) stage is [sig | tau]. sig: this CTA's 64 queries, every column,
    // K-major (HD/64 quadrants of 64 rows x 64 columns): B of S^T (dP^T). tau: the
    // block's 128 queries, this CTA's HD/2 columns, MN-major: B of dK (dV); two
    // 64-row quadrants at d = 128, one 128-row x 32-column box at d = 64.
    static constexpr int kSigBytes = (HD / 64) * kQuad;
    static constexpr int kTauBytes = 128 * HD;                   // 128 rows x HD/2 bf16
    static constexpr int kStageBytes = kSigBytes + kTauBytes;
    static constexpr int kKBytes = 256 * HD;                     // 128 keys x HD bf16
    static constexpr int kKXBytes = 256 * HD;                    // 256 keys x HD/2 bf16
    // bytes per 16 rows along K of an MN-major column half (two 8-row atoms)
    static constexpr uint32_t kMnStep16 = kNarrow ? 1024 : 2048;
    static constexpr int kKOff = 0;                              // own key block, HD/64 boxes
    static constexpr int kVOff = kKOff + kKBytes;
    static constexpr int kKXOff = kVOff + kKBytes;               // K of the pair's 256 keys, this CTA's HD/2 columns
    static constexpr int kQOff = kKXOff + kKXBytes;              // Q ring (stage = dQ staging after dK)
    static constexpr int kDOOff = kQOff + kQStages * kStageBytes;
    static constexpr int kDSOff = kDOOff + kStageBytes;          // dS: 256 key rows x 64 queries
    static constexpr int kDSBytes = 256 * 128;
    static constexpr int kStatOff = kDSOff + kDSBytes;           // per Q stage: -lse2[128], -D[128]
    static constexpr int kBarOff = kStatOff + kQStages * 1024;
    // barriers used on the even CTA only (the pair's MMA waits on them)
    static constexpr int kKVFull = 0, kQFull = 1, kDOFull = kQFull + kQStages, kPFull = kDOFull + 1,
                         kDSFull = kPFull + 1, kDQFree = kDSFull + 1,
                         // barriers of every CTA
                         kKVEmpty = kDQFree + 1, kQEmpty = kKVEmpty + 1, kStatFull = kQEmpty + kQStages,
                         kDOEmpty = kStatFull + kQStages, kSFull = kDOEmpty + 1, kDPFull = kSFull + 1,
                         kDSEmpty = kDPFull + 1, kDQFull = kDSEmpty + 1, kDKVFull = kDQFull + 1,
                         kSemGo = kDKVFull + 1, kRedDone = kSemGo + 1, kDrain = kRedDone + 1,
                         kNumBars = kDrain + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16;
    static constexpr uint32_t kTS = 0, kTDP = 128, kTDV = 256, kTDK = 256 + HD;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(kStageBytes >= 64 * HD * 4, "a Q stage holds the CTA's 64 x HD fp32 dQ tile");
    static_assert(kKXOff % 1024 == 0 && kQOff % 1024 == 0 && kStageBytes % 1024 == 0 && kDSOff % 1024 == 0,
                  "swizzle atoms aligned");
};

struct PairTile {
    int b, h, p;       // batch, key/value head, key-block pair
    int n;             // this CTA's key block (2p + rank)
    int lq, lk;
    int q_row0, k_row0;
    int m_begin, m_end;   // query blocks either key block of the pair sees
    // the tile walks every query head of the group (hq0 .. hq0 + group - 1), each
    // over [m_begin, m_end): step u is query head hq0 + u / nm, block m_begin + u % nm
    int hq0, nm, nblk;
};

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// kSpt (deterministic kernels with a causal mask): pairs walked shortest first,
// so that no tile waits at its first dQ write (FlashAttention-4 paper, Section
// 3.2.4). Without a causal mask every key block sees every query block.
template <bool kSpt>
__device__ __forceinline__ PairTile pair_tile(int t, const BwdParams& p, const VarlenMap* vm, uint32_t rank) {
    const Geometry& g = p.g;
    const bool spt = kSpt && g.causal;
    // heads in L2-sized sections, longest pairs first within a section, where
    // that pays (p.sections, as in bwd.cu); the deterministic kernel keeps one
    // global order of levels, shortest first
    Tile ti = vm ? sched_varlen(*vm, t, g.B, g.Hkv, 2 * kBN, p.head_section, spt, true)
                 : ((g.causal && (spt || !p.sections)) ? sched_dense_lpt(t, g.B, g.Hkv, p.nm, spt)
                                                        : sched_dense(t, g.Hkv, p.nm, p.head_section, false));
    PairTile f;
    f.b = ti.b;
    f.h = ti.h;
    f.p = ti.m;
    f.n = 2 * ti.m + (int)rank;
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
    const int n0 = 2 * ti.m;   // the pair's first key block sees the most query blocks
    f.m_end = (f.lq + kBM - 1) / kBM;
    f.m_begin = g.causal ? max(0, floor_div(n0 * kBN - (f.lk - f.lq), kBM)) : 0;
    if (n0 * kBN >= f.lk || f.m_begin > f.m_end) f.m_begin = f.m_end;
    f.hq0 = f.h * g.group;
    f.nm = f.m_end - f.m_begin;
    f.nblk = g.group * f.nm;
    return f;
}

// Deterministic mode: pairs that add to query block m before pair f.p (from
// the highest pair down with a causal mask, else ascending). The key blocks
// that see query block m are [n_lo, n_hi), so the pairs are [n_lo/2, ceil(n_hi/2)).
__device__ __forceinline__ int pair_dq_turn(const BwdParams& p, const PairTile& f, int m) {
    int n_lo, n_hi;
    band_key_blocks(mask_band(f.lq, f.lk, -1, p.g.causal ? 0 : -1), m * kBM, m * kBM + kBM - 1, kBN, &n_lo, &n_hi);
    return p.g.causal ? (n_hi + 1) / 2 - 1 - f.p : f.p - n_lo / 2;
}

// tmQ64, tmDO64: 64-row x 64-column boxes; tmQ32, tmDO32, tmK32: 128-row x
// 32-column boxes with the 64-byte swizzle (d = 64 only); tmDQ32: the fp32 dQ
// accumulator in 32-row x 32-column boxes.
template <int HD, bool kDet>
__global__ void __launch_bounds__(kThreads, 1)
bwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ64, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO64,
                const __grid_constant__ CUtensorMap tmDQ32, const __grid_constant__ CUtensorMap tmQ32,
                const __grid_constant__ CUtensorMap tmDO32, const __grid_constant__ CUtensorMap tmK32,
                const BwdParams p, const VarlenMap* vm) {
    using Lay = PairLay<HD>;
    constexpr bool kNarrow = Lay::kNarrow;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Geometry& g = p.g;
    const uint32_t rank = cluster_ctarank();
    const bool leader_cta = rank == 0;
    // every CTA takes the same branch here (the shared window is aligned alike)
    if (base & 1023u) {
        if (tid == 0) atomicCAS(p.status, kStatusOk, kStatusMisaligned);
        return;
    }
    auto bar = [&](int i) -> uint32_t { return base + Lay::kBarOff + 8u * (uint32_t)i; };
    // the even CTA's barrier at the same offset (cluster window)
    auto lbar = [&](int i) -> uint32_t { return mapa_shared(bar(i), 0); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kMiscOff + 4);

    if (tid == 0) {
        mbar_init(bar(Lay::kKVFull), 1);
        for (int s = 0; s < Lay::kQStages; ++s) {
            mbar_init(bar(Lay::kQFull + s), 1);
            mbar_init(bar(Lay::kQEmpty + s), 4);   // each dQ warp: its rows of the staged dQ are read
            mbar_init(bar(Lay::kStatFull + s), 1);
        }
        mbar_init(bar(Lay::kDOFull), 1);
        mbar_init(bar(Lay::kPFull), 16);     // 8 compute warps of each CTA
        mbar_init(bar(Lay::kDSFull), 16);
        mbar_init(bar(Lay::kDQFree), 8);     // 4 dQ warps of each CTA
        mbar_init(bar(Lay::kKVEmpty), 1);
        mbar_init(bar(Lay::kDOEmpty), 1);
        mbar_init(bar(Lay::kSFull), 1);
        mbar_init(bar(Lay::kDPFull), 1);
        mbar_init(bar(Lay::kDSEmpty), 1);
        mbar_init(bar(Lay::kDQFull), 1);
        mbar_init(bar(Lay::kDKVFull), 1);
        mbar_init(bar(Lay::kSemGo), 1);
        mbar_init(bar(Lay::kRedDone), 4);      // deterministic: each dQ warp's adds are complete
        mbar_init(bar(Lay::kDrain), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ64);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmDO64);
        tma_prefetch_desc(&tmDQ32);
        if constexpr (kNarrow) {
            tma_prefetch_desc(&tmQ32);
            tma_prefetch_desc(&tmDO32);
            tma_prefetch_desc(&tmK32);
        }
    }
    if (warp == 1) {   // both CTAs allocate: the pair gets the same columns in each
        tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();   // the peer's barriers are initialised before any remote arrival
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{abort_flag, p.status, p.wait_budget_ns};
    const bool varlen = g.cu_seqlens != nullptr;
    const VarlenMap* vmp = varlen ? vm : nullptr;
    const int n_tiles = varlen ? vm->pre[g.B] : p.n_tiles;
    const int cl = (int)cluster_id_x(), ncl = (int)nclusters_x();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        setmaxnreg_dec<kRegsLoadMma>();
        uint32_t tile_it = 0, qc = 0;
        bool ok = true;
        float* stats = reinterpret_cast<float*>(smem + Lay::kStatOff);
        // one Q (dO) stage of query block rows [qrow, qrow + 128): sig = this CTA's
        // 64 queries, every column; tau = the 128 queries, this CTA's HD/2 columns
        auto load_stage = [&](uint32_t dst, const CUtensorMap* m64, const CUtensorMap* m32, uint32_t full, int hq,
                              int qrow) {
            for (int c = 0; c < HD / 64; ++c)
                tma_load_3d_pair(dst + c * kQuad, m64, full, c * 64, hq, qrow + 64 * (int)rank);
            if constexpr (kNarrow) {
                tma_load_3d_pair(dst + Lay::kSigBytes, m32, full, 32 * (int)rank, hq, qrow);
            } else {
                tma_load_3d_pair(dst + Lay::kSigBytes, m64, full, 64 * (int)rank, hq, qrow);
                tma_load_3d_pair(dst + Lay::kSigBytes + kQuad, m64, full, 64 * (int)rank, hq, qrow + 64);
            }
        };
        for (int k = 0, t = cl; t < n_tiles && ok; t = snake_tile(cl, ++k, ncl)) {
            const PairTile f = pair_tile<kDet>(t, p, vmp, rank);
            if (f.m_begin >= f.m_end) continue;
            ok = warp_wait_cluster(bar(Lay::kKVEmpty), (tile_it & 1u) ^ 1u, w, lane);
            if (!ok) break;
            if (lane == 0) {
                const uint32_t full = lbar(Lay::kKVFull);
                // K, V, KX of both CTAs
                if (leader_cta) mbar_expect_tx(bar(Lay::kKVFull), 2u * (2u * Lay::kKBytes + Lay::kKXBytes));
                const int krow = f.k_row0 + f.n * kBN, krow0 = f.k_row0 + 2 * f.p * kBN;
                for (int c = 0; c < HD / 64; ++c) {
                    tma_load_3d_pair(base + Lay::kKOff + c * kBox, &tmK, full, c * 64, f.h, krow);
                    tma_load_3d_pair(base + Lay::kVOff + c * kBox, &tmV, full, c * 64, f.h, krow);
                }
                // the pair's 256 keys, this CTA's HD/2 columns of K (B of the dQ product)
                for (int hf = 0; hf < 2; ++hf) {
                    if constexpr (kNarrow)
                        tma_load_3d_pair(base + Lay::kKXOff + hf * (Lay::kKXBytes / 2), &tmK32, full, (int)rank * 32,
                                         f.h, krow0 + hf * kBN);
                    else
                        tma_load_3d_pair(base + Lay::kKXOff + hf * kBox, &tmK, full, (int)rank * 64, f.h,
                                         krow0 + hf * kBN);
                }
            }
            __syncwarp();
            ++tile_it;
            for (int u = 0; u < f.nblk && ok; ++u) {
                const int hq = f.hq0 + u / f.nm, m = f.m_begin + u % f.nm;
                const uint32_t st = qc % Lay::kQStages;
                ok = warp_wait(bar(Lay::kQEmpty + st), ((qc / Lay::kQStages) & 1u) ^ 1u, w, lane);
                if (!ok) break;
                const int qrow = f.q_row0 + m * kBM;
                if (lane == 0) {
                    const uint32_t full = lbar(Lay::kQFull + st), dst = base + Lay::kQOff + st * Lay::kStageBytes;
                    if (leader_cta) mbar_expect_tx(bar(Lay::kQFull + st), 2u * Lay::kStageBytes);
                    load_stage(dst, &tmQ64, &tmQ32, full, hq, qrow);
                }
                // row statistics of the query block, negated: -lse (log2 units), -D
                float* nlse2 = stats + st * 256;
                float* ndd = nlse2 + 128;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = m * kBM + lane * 4 + e;
                    float lv = -INFINITY, dv = 0.f;
                    if (r < f.lq) {
                        const long si = varlen ? (long)hq * g.Lq + f.q_row0 + r : ((long)f.b * g.H + hq) * g.Lq + r;
                        lv = -p.lse[si] * kLog2e;
                        dv = -p.delta[si];
                    }
                    nlse2[lane * 4 + e] = lv;
                    ndd[lane * 4 + e] = dv;
                }
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Lay::kStatFull + st));
                ok = warp_wait_cluster(bar(Lay::kDOEmpty), (qc & 1u) ^ 1u, w, lane);
                if (!ok) break;
                if (lane == 0) {
                    const uint32_t full = lbar(Lay::kDOFull), dst = base + Lay::kDOOff;
                    if (leader_cta) mbar_expect_tx(bar(Lay::kDOFull), 2u * Lay::kStageBytes);
                    load_stage(dst, &tmDO64, &tmDO32, full, hq, qrow);
                }
                __syncwarp();
                ++qc;
            }
        }
        // the even CTA drains the pair's copies (their completions count on its barriers)
        if (lane == 0 && leader_cta) {
            if (tile_it) drain_wait(bar(Lay::kKVFull), (tile_it - 1) & 1u, p.wait_budget_ns);
            for (uint32_t i = 0; i < (uint32_t)Lay::kQStages && i < qc; ++i) {
                const uint32_t n = qc - 1 - i;
                drain_wait(bar(Lay::kQFull + n % Lay::kQStages), (n / Lay::kQStages) & 1u, p.wait_budget_ns);
            }
            if (qc) drain_wait(bar(Lay::kDOFull), (qc - 1) & 1u, p.wait_budget_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        setmaxnreg_dec<kRegsLoadMma>();
        if (leader_cta) {
            constexpr uint32_t kIdS = idesc_bf16_f32(2 * kBN, kBM, false, false);   // S^T, dP^T: 256 x 128
            constexpr uint32_t kIdKV = idesc_bf16_f32(2 * kBN, HD, false, true);    // dV, dK: 256 x d
            constexpr uint32_t kIdDQ = idesc_bf16_f32(kBM, HD, true, true);         // dQ: 128 x d
            const SmemDesc k_km = sdesc_sw128_split(base + Lay::kKOff, 16, 1024);
            const SmemDesc v_km = sdesc_sw128_split(base + Lay::kVOff, 16, 1024);
            // MN-major column halves: 64-byte swizzle at d = 64, 128-byte at d = 128
            auto mn_half = [&](uint32_t off) {
                return kNarrow ? sdesc_sw64_split(base + off, 16384, 512) : sdesc_sw128_split(base + off, kBox, 1024);
            };
            const SmemDesc kx_mn = mn_half(Lay::kKXOff);
            const SmemDesc ds_mn = sdesc_sw128_split(base + Lay::kDSOff, kBox, 1024);
            const SmemDesc q_km0 = sdesc_sw128_split(base + Lay::kQOff, 16, 1024);
            const SmemDesc q_mn0 = mn_half(Lay::kQOff + Lay::kSigBytes);
            const SmemDesc do_km = sdesc_sw128_split(base + Lay::kDOOff, 16, 1024);
            const SmemDesc do_mn = mn_half(Lay::kDOOff + Lay::kSigBytes);
            auto at_stage = [&](SmemDesc d, uint32_t stage) {
                d.lo += stage * desc_step(Lay::kStageBytes);
                return d;
            };
            // D[256 x 128] = A[256 x d] * B[128 x d]^T: A K-major in 64-column boxes of
            // 128 rows, B K-major in 64-column quadrants of this CTA's 64 rows
            auto mma_nt = [&](uint32_t d_tmem, SmemDesc a, SmemDesc b) {
#pragma unroll
                for (int k = 0; k < HD / 16; ++k)
                    mma_pair_ss(d_tmem, a, desc_step((k >> 2) * kBox + (k & 3) * 32), b,
                                desc_step((k >> 2) * kQuad + (k & 3) * 32), kIdS, k > 0);
            };
            uint32_t tile_it = 0, qc = 0, pc = 0, dsc = 0, dqf = 0;
            bool ok = true;
            for (int k = 0, t = cl; t < n_tiles && ok; t = snake_tile(cl, ++k, ncl)) {
                const PairTile f = pair_tile<kDet>(t, p, vmp, rank);
                if (f.m_begin >= f.m_end) continue;
                const int nblk = f.nblk;
                ok = warp_wait_cluster(bar(Lay::kKVFull), tile_it & 1u, w, lane);
                if (!ok) break;
                ++tile_it;
                uint32_t st = qc % Lay::kQStages;
                ok = warp_wait_cluster(bar(Lay::kQFull + st), (qc / Lay::kQStages) & 1u, w, lane);
                if (!ok) break;
                tc_fence_after_sync();
                if (lane == 0) {
                    mma_nt(tmem + Lay::kTS, k_km, at_stage(q_km0, st));
                    tc_commit_pair(bar(Lay::kSFull), 3);
                }
                __syncwarp();
                for (int u = 0; u < nblk; ++u) {
                    const SmemDesc q_mn = at_stage(q_mn0, st);
                    ok = warp_wait_cluster(bar(Lay::kDQFree), (dqf & 1u) ^ 1u, w, lane);
                    if (!ok) break;
                    ++dqf;
                    ok = warp_wait_cluster(bar(Lay::kDOFull), qc & 1u, w, lane);
                    if (!ok) break;
                    tc_fence_after_sync();
                    if (lane == 0) {
                        mma_nt(tmem + Lay::kTDP, v_km, do_km);
                        tc_commit_pair(bar(Lay::kDPFull), 3);
                    }
                    __syncwarp();
                    ok = warp_wait_cluster(bar(Lay::kPFull), pc & 1u, w, lane);
                    if (!ok) break;
                    ++pc;
                    tc_fence_after_sync();
                    if (lane == 0) {
#pragma unroll
                        for (int kk = 0; kk < kBM / 16; ++kk)
                            mma_pair_ts(tmem + Lay::kTDV, tmem + Lay::kTS + packed_col(kk), do_mn,
                                        desc_step(kk * Lay::kMnStep16), kIdKV, (u > 0 || kk > 0) ? 1u : 0u);
                        tc_commit_pair(bar(Lay::kDOEmpty), 3);
                    }
                    __syncwarp();
                    const bool more = u + 1 < nblk;
                    const uint32_t st_next = more ? (qc + 1) % Lay::kQStages : st;
                    if (more) {   // next query block's S^T right after dV (it overwrites the consumed P^T)
                        ok = warp_wait_cluster(bar(Lay::kQFull + st_next), ((qc + 1) / Lay::kQStages) & 1u, w, lane);
                        if (!ok) break;
                        tc_fence_after_sync();
                        if (lane == 0) {
                            mma_nt(tmem + Lay::kTS, k_km, at_stage(q_km0, st_next));
                            tc_commit_pair(bar(Lay::kSFull), 3);
                        }
                        __syncwarp();
                    }
                    ok = warp_wait_cluster(bar(Lay::kDSFull), dsc & 1u, w, lane);
                    if (!ok) break;
                    ++dsc;
                    tc_fence_after_sync();
                    if (lane == 0) {
#pragma unroll
                        for (int kk = 0; kk < kBM / 16; ++kk)
                            mma_pair_ts(tmem + Lay::kTDK, tmem + Lay::kTDP + packed_col(kk), q_mn,
                                        desc_step(kk * Lay::kMnStep16), kIdKV, (u > 0 || kk > 0) ? 1u : 0u);
                        // dQ over the pair's 256 keys: key rows 0-127 are the even CTA's block
#pragma unroll
                        for (int kk = 0; kk < 2 * kBN / 16; ++kk)
                            mma_pair_ss(tmem + Lay::kTDP, ds_mn, desc_step(kk * 2048), kx_mn,
                                        desc_step(kk * Lay::kMnStep16), kIdDQ, kk > 0 ? 1u : 0u);
                        tc_commit_pair(bar(Lay::kDQFull), 3);
                        tc_commit_pair(bar(Lay::kDSEmpty), 3);
                        if (!more) {
                            tc_commit_pair(bar(Lay::kDKVFull), 3);
                            tc_commit_pair(bar(Lay::kKVEmpty), 3);
                        }
                    }
                    __syncwarp();
                    ++qc;
                    st = st_next;
                }
            }
            if (lane == 0) {
                tc_commit_pair(bar(Lay::kDrain), 1);
                drain_wait(bar(Lay::kDrain), 0, p.wait_budget_ns);
            }
            __syncwarp();
        }
    } else if (warp < 4) {
        setmaxnreg_dec<kRegsLoadMma>();
    } else if (warp < 12) {
        // ------------------------------------------------------------ compute warpgroups (both CTAs)
        const int wg = (warp - 4) >> 2;            // query columns [64 wg, 64 wg + 64)
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;         // key row inside this CTA's block
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = g.scale_log2;
        const float* stats = reinterpret_cast<const float*>(smem + Lay::kStatOff);
        // dS of query half wg goes to CTA wg, key rows 128 rank + r of its dS tile
        const uint32_t ds_row = mapa_shared(base + Lay::kDSOff, (uint32_t)wg) +
                                (uint32_t)(((128 * (int)rank + r) >> 3) * 1024 + (r & 7) * 128);
        const uint32_t pfull = lbar(Lay::kPFull), dsfull = lbar(Lay::kDSFull);
        uint32_t sc = 0, qc = 0, dpc = 0, dse = 0, tile_it = 0;
        bool ok = true;
        uint32_t rr[32];
        for (int k = 0, t = cl; t < n_tiles && ok; t = snake_tile(cl, ++k, ncl)) {
            const PairTile f = pair_tile<kDet>(t, p, vmp, rank);
            const int key = f.n * kBN + r;
            const bool key_ok = key < f.lk;
            const long kv_off = (((long)f.k_row0 + key) * g.Hkv + f.h) * HD + wg * (HD / 2);
            if (f.nblk == 0) {   // no query sees the pair's keys
                if (key_ok) {
#pragma unroll
                    for (int c = 0; c < HD / 16; ++c) {
                        reinterpret_cast<uint4*>(p.dv + kv_off)[c] = make_uint4(0, 0, 0, 0);
                        reinterpret_cast<uint4*>(p.dk + kv_off)[c] = make_uint4(0, 0, 0, 0);
                    }
                }
                continue;
            }
            // query q is allowed for this key iff q_lo <= q < q_hi; a key past the
            // sequence (the pair's odd block at its end) sees none
            const int q_lo = key_ok ? (g.causal ? key - (f.lk - f.lq) : 0) : f.lq;
            const int q_hi = f.lq;
            for (int u = 0; u < f.nblk; ++u) {
                const int m = f.m_begin + u % f.nm;
                const uint32_t st = qc % Lay::kQStages;
                ok = warp_wait_cluster(bar(Lay::kSFull), sc & 1u, w, lane);
                if (!ok) break;
                ++sc;
                ok = warp_wait(bar(Lay::kStatFull + st), (qc / Lay::kQStages) & 1u, w, lane);
                if (!ok) break;
                ++qc;
                tc_fence_after_sync();
                float pv[64];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    tmem_ld32(tmem + lane_off + Lay::kTS + wg * 64 + c * 32, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) pv[c * 32 + i] = u2f(rr[i]);
                }
                const float* nlse2 = stats + st * 256 + wg * 64;
                const float* ndd = stats + st * 256 + 128 + wg * 64;
                const int q0 = m * kBM + wg * 64;
                const bool full = q0 >= q_lo && q0 + 64 <= q_hi;
                const uint64_t sc2 = f32x2(sl2, sl2);
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const float2 nl = *reinterpret_cast<const float2*>(nlse2 + c);
                    float x0, x1;
                    f32x2_split(ffma2(f32x2(pv[c], pv[c + 1]), sc2, f32x2(nl.x, nl.y)), x0, x1);
                    pv[c] = ex2_mufu(x0);
                    pv[c + 1] = ex2_mufu(x1);
                }
                if (!full) {
                    const int lo = q_lo - q0, hi = q_hi - q0;
#pragma unroll
                    for (int c = 0; c < 64; ++c) pv[c] = (c >= lo && c < hi) ? pv[c] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) rr[i] = pack_bf16x2(pv[2 * i], pv[2 * i + 1]);
                tmem_st32(tmem + lane_off + Lay::kTS + wg * 64, rr);
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(pfull);
                // dS^T = P^T * (dP^T - D)
                ok = warp_wait_cluster(bar(Lay::kDPFull), dpc & 1u, w, lane);
                if (!ok) break;
                ++dpc;
                tc_fence_after_sync();
                ok = warp_wait_cluster(bar(Lay::kDSEmpty), (dse & 1u) ^ 1u, w, lane);
                if (!ok) break;
                ++dse;
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
                                              fadd2(f32x2(u2f(rr[i + 2 * e]), u2f(rr[i + 2 * e + 1])),
                                                    f32x2(nd.x, nd.y))),
                                        d0, d1);
                            ds2[cc >> 1] = pack_bf16x2(d0, d1);
                        }
                        // 128-byte swizzle: 16-byte chunk j of row x lands at chunk j ^ (x % 8)
                        const int chunk = (c * 32 + i) >> 3;
                        const int b = (c * 32 + i) >> 1;
                        st_cluster_v4(ds_row + (uint32_t)((chunk ^ (r & 7)) << 4),
                                      make_uint4(ds2[b], ds2[b + 1], ds2[b + 2], ds2[b + 3]));
                    }
                }
                // dS^T also into tensor memory (this warpgroup's dP^T columns, already read) for dK
                tmem_st32(tmem + lane_off + Lay::kTDP + wg * 64, ds2);
                fence_proxy_async_smem_cluster();
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(dsfull);
            }
            if (!ok) break;
            // epilogue: this warpgroup writes d/2 columns of dV and of dK for its key row
            ok = warp_wait_cluster(bar(Lay::kDKVFull), tile_it & 1u, w, lane);
            if (!ok) break;
            ++tile_it;
            tc_fence_after_sync();
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t col0 = (which ? Lay::kTDK : Lay::kTDV) + wg * (HD / 2);
                const float mul = which ? g.scale : 1.f;
                __nv_bfloat16* dst = (which ? p.dk : p.dv) + kv_off;
#pragma unroll
                for (int c = 0; c < HD / 64; ++c) {
                    tmem_ld32(tmem + lane_off + col0 + c * 32, rr);
                    if (key_ok) {
                        uint32_t o2[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            o2[i] = pack_bf16x2(u2f(rr[2 * i]) * mul, u2f(rr[2 * i + 1]) * mul);
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
        // ------------------------------------------------------------ dQ warpgroup (both CTAs)
        // This CTA's 64 queries of the block x HD columns, summed over the pair's
        // 256 keys by the MMA: tensor-memory lanes 0-63 hold columns 0 .. HD/2-1 of
        // query rows 0-63 and lanes 64-127 columns HD/2 .. HD-1 of the same rows.
        // Staged through the Q stage the block's dK product has finished reading, as
        // HD/32 64-row x 32-column swizzled boxes; each warp adds its own 32 rows x
        // HD/2 columns with TMA reduce-adds issued by its lane 0. Deterministic
        // mode: under the semaphore of this query-row half, pairs in a fixed order,
        // every warp's adds complete before the next pair's turn.
        const int q4 = warp - 12;
        const int qr = (q4 & 1) * 32 + lane;      // query row inside this CTA's 64
        const int half = q4 >> 1;                 // columns [HD/2 half, HD/2 half + HD/2)
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        setmaxnreg_inc<kRegsDq>();
        const bool leader = warp == 12 && lane == 0;
        const uint32_t dqfree = lbar(Lay::kDQFree);
        uint32_t dqc = 0, sgo = 0, rdc = 0;
        bool ok = true;
        uint32_t rr[32];
        for (int k = 0, t = cl; t < n_tiles && ok; t = snake_tile(cl, ++k, ncl)) {
            const PairTile f = pair_tile<kDet>(t, p, vmp, rank);
            for (int u = 0; u < f.nblk; ++u) {
                const int hq = f.hq0 + u / f.nm, m = f.m_begin + u % f.nm;
                const uint32_t st = dqc % Lay::kQStages;
                ok = warp_wait_cluster(bar(Lay::kDQFull), dqc & 1u, w, lane);
                if (!ok) break;
                ++dqc;
                tc_fence_after_sync();
                int* sem = nullptr;
                if constexpr (kDet) {
                    const long tile = varlen ? (long)hq * (g.Lq / kBM + g.B + 1) + f.q_row0 / kBM + f.b + m
                                             : ((long)f.b * g.H + hq) * p.nq + m;
                    sem = p.semaphores + 2 * tile + rank;
                    if (leader) {
                        if (sem_wait(sem, pair_dq_turn(p, f, m), w)) fence_proxy_async_global();
                        mbar_arrive(bar(Lay::kSemGo));   // arrive even after a failure; abort_flag tells
                    }
                    ok = warp_wait(bar(Lay::kSemGo), sgo & 1u, w, lane);
                    ++sgo;
                    ok = ok && !*abort_flag;
                    if (!ok) break;
                }
                uint32_t row[HD / 2];
#pragma unroll
                for (int c = 0; c < HD / 64; ++c) {
                    tmem_ld32(tmem + lane_off + Lay::kTDP + c * 32, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) row[c * 32 + i] = rr[i];
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(dqfree);
                uint8_t* stage = smem + Lay::kQOff + st * Lay::kStageBytes;
                const uint32_t stage_s = base + Lay::kQOff + st * Lay::kStageBytes;
#pragma unroll
                for (int bx = 0; bx < HD / 64; ++bx) {   // this half's boxes: 32 columns each
                    uint8_t* srow = stage + ((HD / 64) * half + bx) * kQuad + (qr >> 3) * 1024 + (qr & 7) * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4*>(srow + ((j ^ (qr & 7)) << 4)) =
                            make_uint4(row[bx * 32 + 4 * j], row[bx * 32 + 4 * j + 1], row[bx * 32 + 4 * j + 2],
                                       row[bx * 32 + 4 * j + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // this warp's 32 rows (rows past the sequence carry exact zeros: P = 0 there)
                    for (int bx = 0; bx < HD / 64; ++bx) {
                        const int box = (HD / 64) * half + bx;
                        tma_reduce_add_3d(&tmDQ32, stage_s + box * kQuad + (q4 & 1) * 4096, box * 32, hq,
                                          f.q_row0 + m * kBM + 64 * (int)rank + (q4 & 1) * 32);
                    }
                    bulk_commit_group();
                    if constexpr (kDet) {
                        bulk_wait_group0();
                        fence_proxy_async_global();
                        mbar_arrive(bar(Lay::kRedDone));
                    } else {
                        bulk_wait_group_read0();
                    }
                    mbar_arrive(bar(Lay::kQEmpty + st));   // this warp's rows of the stage are read
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
    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();   // the even CTA's MMAs, which read both CTAs, are complete
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
    cluster_sync_all();
}

}  // namespace

bool bwd_pair_supported(const BwdParams& p) {
    const Geometry& g = p.g;
    return (g.d == 64 || g.d == 128) && p.d_v == g.d && g.win_left < 0 && (g.win_right < 0 || g.win_right == 0) &&
           p.mask.ptr == nullptr;
}

int bwd_pair_tiles_per_head(int Lk) { return (Lk + 2 * kBN - 1) / (2 * kBN); }

namespace {

template <int HD>
cudaError_t launch_pair_hd(const PairMaps& pm, const CUtensorMap& tk, const CUtensorMap& tv, const BwdParams& p,
                           const void* varlen_map, int num_sms, cudaStream_t stream) {
    using Lay = PairLay<HD>;
    auto kern = p.deterministic ? bwd_pair_kernel<HD, true> : bwd_pair_kernel<HD, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // every cluster must be resident at once: the deterministic mode's waits on
    // other clusters' dQ turns assume it
    cfg.gridDim = dim3(2 * (num_sms / 2));
    int max_clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const bool varlen = p.g.cu_seqlens != nullptr;
    const int clusters = varlen ? max_clusters : min(p.n_tiles, max_clusters);
    if (clusters <= 0) return cudaSuccess;
    cfg.gridDim = dim3(2 * clusters);
    return cudaLaunchKernelEx(&cfg, kern, pm.q64, tk, tv, pm.do64, pm.dq32, pm.q32, pm.do32, pm.k32, p,
                              static_cast<const VarlenMap*>(varlen_map));
}

}  // namespace

cudaError_t launch_bwd_pair(const PairMaps& pm, const CUtensorMap& tk, const CUtensorMap& tv, const BwdParams& p,
                            const void* varlen_map, int num_sms, cudaStream_t stream) {
    switch (p.g.d) {
        case 64: return launch_pair_hd<64>(pm, tk, tv, p, varlen_map, num_sms, stream);
        case 128: return launch_pair_hd<128>(pm, tk, tv, p, varlen_map, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
