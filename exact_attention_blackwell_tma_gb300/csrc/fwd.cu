// Forward kernel: O = softmax(scale * Q K^T [+ causal mask]) V and the row
// log-sum-exp, tile by tile, with the score tile S kept in tensor memory.
//
// Design (FlashAttention-4 paper, Section 3.1.2 "New pipeline for overlapping
// MMA and softmax", Section 3.1.4 "Skipping online softmax rescaling"; blog
// post on FA4, "Tile life cycle" and "Warp specialisation"):
//  * each work tile is two 128-row Q tiles of one (batch, head); the MMA of one
//    tile overlaps the softmax of the other (ping-pong);
//  * warp roles: warp 0 issues TMA loads (Q once per tile, K/V blocks through
//    a ring of shared-memory stages), warp 1 issues tcgen05 MMAs (from one
//    thread; at d = 64 one elected lane of the converged warp), warps 4-7 and
//    8-11 are the two softmax warpgroups (one query row per thread, so the row
//    max needs no shuffles);
//  * tensor memory holds S_0, S_1 (fp32, 128 columns each) and O_0, O_1
//    (fp32, d columns each); P is written as bf16 over the first half of its
//    S tile and read by the PV MMA straight from tensor memory. At d = 64, P
//    has 64 columns of its own per Q tile (the columns d = 128 needs for O):
//    the next block's S is computed as soon as the softmax has loaded the
//    current one, and the MMAs are issued by the converged warp (B2 H16 L8192
//    d64: causal 642 -> 758 TF/s, non-causal 679 -> 823);
//  * the running max is only moved when it grows by more than kTau (log2
//    units); the decision is warp-uniform (if any row of a warp needs it, the
//    warp rescales). Results are unchanged because the final normalisation
//    uses the same stale max for the sum and the output.
// Every wait is bounded (see ptx.cuh); on a timeout the kernel records an
// error, stops issuing work, waits (bounded) for its own copies and MMAs in
// flight, frees its tensor memory and returns.
#include "kernels.h"
#include "ptx.cuh"
#include "mask.cuh"
#include "sched.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;            // query rows per Q tile
constexpr int kBN = 128;            // keys per K/V block
constexpr int kRowsPerTile = 2 * kBM;
constexpr int kThreads = 384;       // 12 warps
constexpr float kTau = 8.0f;        // rescale threshold, log2 units (a factor of 256)
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 16384;         // one 128-row x 64-column bf16 TMA box
// Register split: the kernel is compiled for 168 registers per thread
// (384 threads, one CTA per SM); the load/MMA warpgroup gives registers up
// and the two softmax warpgroups, which hold a 128-column score row each,
// take them.
constexpr int kLaunchRegs = 168;
constexpr uint32_t kRegsLoadMma = 88, kRegsSoftmax = 208;
static_assert((kRegsLoadMma + 2 * kRegsSoftmax) * 128 <= kLaunchRegs * kThreads, "register split");

template <int HD>
struct FwdLayout {
    static constexpr int kHalves = HD / 64;             // 64-column boxes per row
    static constexpr int kTileBytes = kBM * HD * 2;     // one 128 x HD bf16 tile
    static constexpr int kStages = HD == 64 ? 8 : 4;    // K/V ring depth (tiles)
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = 2 * kTileBytes;
    static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
    // barrier indices
    static constexpr int kQFull = 0, kQEmpty = 1, kKVFull = 2, kKVEmpty = 2 + kStages,
                         kSFull = 2 + 2 * kStages, kPFull = kSFull + 2, kOFull = kPFull + 2,
                         kDrain = kOFull + 2, kSFree = kDrain + 1, kPVDone = kSFree + 2, kNumBars = kPVDone + 2;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;          // tmem base, abort flag
    static constexpr int kMapOff = (kMiscOff + 16 + 15) / 16 * 16;
    static constexpr int kSmemBytes = kMapOff + (int)sizeof(VarlenMap) + 1024;  // + alignment slack
    static constexpr uint32_t kTmemO0 = 256, kTmemO1 = 256 + HD;
    // d = 64 leaves 128 columns free: each Q tile's bf16 P gets 64 of its own
    // (kSepP), so the next S can be computed while the softmax still works on
    // the current block; at d = 128, P is written over the S it came from.
    static constexpr bool kSepP = HD == 64;
    static constexpr uint32_t kTmemP0 = kSepP ? 384 : 0, kTmemP1 = kSepP ? 448 : 128;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(256 + 2 * HD + (kSepP ? 128 : 0) <= (int)kTmemCols, "tensor memory budget");
};

// Partial exp2 emulation (FlashAttention-4 paper, Section 3.1.3): with kPoly > 0,
// one pair of score columns in every kPoly is exponentiated by the FMA
// polynomial instead of the MUFU unit (kPoly = 8: 12.5% of the entries, 4: 25%;
// the paper emulates 10-25%), never on a row's last K/V block (FA4 blog,
// "关键实现技术"). kPoly = 0: MUFU only. The launcher picks the kernel from the
// per-head-dim setting of attn_set_exp2_emulation.
//
// P = 2^(s * sl2 - m) for one 128-column row, packed to bf16 pairs into tensor
// memory at t_p (64 columns); the fp32 sum goes to l0 + l1.
template <int kPoly>
__device__ __forceinline__ void exp_row_to_tmem(const float (&s)[128], float sl2, float neg_m, uint32_t t_p,
                                                float& l0, float& l1) {
    // x = s * sl2 - m and the running sum on packed fp32 pairs: half the FMA/add
    // instructions of the per-element form (the exp phase is bound by instruction
    // issue; this measured 4-5% faster)
    const uint64_t sc2 = f32x2(sl2, sl2), nm2 = f32x2(neg_m, neg_m);
    uint64_t acc_a = f32x2(0.f, 0.f), acc_b = acc_a;
    uint32_t rr[32];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {   // P columns [32*hf, 32*hf+32) hold keys [64*hf, 64*hf+64)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float x0, x1;
            f32x2_split(ffma2(f32x2(s[64 * hf + 2 * i], s[64 * hf + 2 * i + 1]), sc2, nm2), x0, x1);
            const bool poly = kPoly > 0 && (i % (kPoly > 0 ? kPoly : 1)) == kPoly - 1;
            const float p0 = poly ? ex2_poly3(x0) : ex2_mufu(x0);
            const float p1 = poly ? ex2_poly3(x1) : ex2_mufu(x1);
            if (i & 1) acc_b = fadd2(acc_b, f32x2(p0, p1));
            else acc_a = fadd2(acc_a, f32x2(p0, p1));
            rr[i] = pack_bf16x2(p0, p1);
        }
        tmem_st32(t_p + 32 * hf, rr);
    }
    float a0, a1;
    f32x2_split(fadd2(acc_a, acc_b), a0, a1);
    l0 += a0;
    l1 += a1;
}

struct FwdTile {
    int b, h, mp;      // batch, query head, 256-row query block
    int hk;            // key/value head read by query head h
    int lq, lk;        // sequence lengths
    int q_row0;        // packed row of the first query row of the tile
    int k_row0;        // packed row of the first key of the sequence
    // The tile streams K/V blocks kv_first .. kv_first + n_kv - 1 (n_kv = 0: no
    // row of the tile sees a key). Q tile 0 visits stream blocks [0, n_kv0),
    // Q tile 1 [kv_start1, n_kv): the two tiles' key ranges, 128 rows apart,
    // differ by at most a block at either end (the causal diagonal, a local
    // window's left edge); n_kv0 = 0 when none of tile 0's rows sees a key.
    int kv_first, n_kv, n_kv0, kv_start1;
    // block-sparse (block mask given): the stream is the blocks in
    // [kv_first, kb_end) active in either Q tile's mask row (mrow1 null: tile
    // 1 has no row block); both Q tiles walk all of it (n_kv0 = n_kv,
    // kv_start1 = 0) and mask the blocks their own row drops
    const unsigned char* mrow0;
    const unsigned char* mrow1;
    int kb_end;
};

// kGeneral: the mask has a left bound (a local window) or a block mask.
// Without either every row's keys start at key 0 and every block in range is
// visited, so the kernels instantiated with kGeneral = false keep the stream
// start, Q tile 1's first block and the rows' lower column bound at the
// constant 0 and contain no mask scans (fewer live registers in the softmax
// loop). kSparse (with kGeneral only): a block mask is given. lane: the
// calling warp's lane (the block-mask scans are warp-wide).
template <bool kGeneral, bool kSparse>
__device__ __forceinline__ FwdTile fwd_tile(int t, const FwdParams& p, const VarlenMap& vm, bool varlen, int lane) {
    const Geometry& g = p.g;
    Tile ti = varlen ? sched_varlen(vm, t, g.B, g.H, kRowsPerTile, p.head_section, g.causal != 0, false)
                     : (g.causal ? sched_dense_lpt(t, g.B, g.H, p.nm, true) : sched_dense(t, g.H, p.nm, p.head_section, false));
    FwdTile f;
    f.b = ti.b;
    f.h = ti.h;
    f.hk = ti.h / g.group;
    f.mp = ti.m;
    if (varlen) {
        f.lq = vm_lq(vm, ti.b);
        f.lk = vm_lk(vm, ti.b);
        f.q_row0 = vm.start[ti.b] + ti.m * kRowsPerTile;
        f.k_row0 = vm.start_k[ti.b];
    } else {
        f.lq = g.Lq;
        f.lk = g.Lk;
        f.q_row0 = ti.b * g.Lq + ti.m * kRowsPerTile;
        f.k_row0 = ti.b * g.Lk;
    }
    const MaskBand mb = mask_band(f.lq, f.lk, g.win_left, g.win_right);
    const int r0 = ti.m * kRowsPerTile;
    int l0, h0, l1, h1;
    const bool has0 = band_key_blocks(mb, r0, r0 + kBM - 1, kBN, &l0, &h0);
    bool has1 = band_key_blocks(mb, r0 + kBM, r0 + kRowsPerTile - 1, kBN, &l1, &h1);
    if (!has1 && has0) {   // tile 1 has no row in the sequence: it shadows tile 0 (rows not stored)
        l1 = l0;
        h1 = h0;
        has1 = true;
    }
    // (tile 1's rows follow tile 0's, so with both present l0 <= l1 and h0 <= h1;
    // tile 1 sees no key only if tile 0 sees none either)
    f.kv_first = kGeneral ? (has0 ? l0 : l1) : 0;
    f.n_kv = has1 ? h1 - f.kv_first : 0;
    f.n_kv0 = has0 ? h0 - f.kv_first : 0;
    f.kv_start1 = kGeneral && has1 ? l1 - f.kv_first : 0;
    f.mrow0 = f.mrow1 = nullptr;
    f.kb_end = f.kv_first + f.n_kv;
    if constexpr (kSparse) {
        if (p.mask.ptr) {
            const int mh = p.mask.heads == 1 ? 0 : ti.h, qb = 2 * ti.m;
            f.mrow0 = p.mask.ptr + ((long)mh * mask_rows(g) + qb) * mask_cols(g);
            f.mrow1 = qb + 1 < mask_rows(g) ? f.mrow0 + mask_cols(g) : nullptr;
            f.n_kv = f.n_kv > 0 ? sparse_count(f.mrow0, f.mrow1, f.kv_first, f.kb_end, lane) : 0;
            f.n_kv0 = f.n_kv;
            f.kv_start1 = 0;
        }
    }
    return f;
}

template <int HD, bool kGeneral, bool kSparse, int kPoly>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using Lay = FwdLayout<HD>;
    constexpr int S = Lay::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Geometry& g = p.g;
    const bool varlen = g.cu_seqlens != nullptr;

    auto bar = [&](int i) -> uint32_t { return base + Lay::kBarOff + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kMiscOff + 4);
    VarlenMap& vm = *reinterpret_cast<VarlenMap*>(smem + Lay::kMapOff);

    if (tid == 0) {
        mbar_init(bar(Lay::kQFull), 1);
        mbar_init(bar(Lay::kQEmpty), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(Lay::kKVFull + s), 1);
            mbar_init(bar(Lay::kKVEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(Lay::kSFull + t), 1);
            mbar_init(bar(Lay::kPFull + t), 4 * 32);
            mbar_init(bar(Lay::kOFull + t), 1);
            mbar_init(bar(Lay::kSFree + t), 4 * 32);   // (d = 64) the softmax has read its S
            mbar_init(bar(Lay::kPVDone + t), 1);       // (d = 64) PV has read P and added into O
        }
        mbar_init(bar(Lay::kDrain), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    int n_tiles = p.n_tiles;
    if (varlen) {
        sched_varlen_build(vm, g.cu_seqlens, g.cu_seqlens_k, g.B, g.H, kRowsPerTile, false, tid, kThreads);
        n_tiles = vm.pre[g.B];
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{abort_flag, p.status, p.wait_budget_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        setmaxnreg_dec<kRegsLoadMma>();
        uint32_t kv_cnt = 0, it = 0, q_issued = 0;
        bool ok = true;
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const FwdTile f = fwd_tile<kGeneral, kSparse>(t, p, vm, varlen, lane);
            if (f.n_kv == 0) continue;
            ok = warp_wait(bar(Lay::kQEmpty), (it & 1u) ^ 1u, w, lane);
            if (!ok) break;
            if (lane == 0) {
                mbar_expect_tx(bar(Lay::kQFull), 2 * Lay::kTileBytes);
                for (int tq = 0; tq < 2; ++tq)
                    for (int hf = 0; hf < Lay::kHalves; ++hf)
                        tma_load_3d(base + Lay::kQOff + tq * Lay::kTileBytes + hf * kBox, &tmQ,
                                    bar(Lay::kQFull), hf * 64, f.h, f.q_row0 + tq * kBM);
            }
            __syncwarp();
            ++q_issued;
            const bool sparse = kSparse && f.mrow0 != nullptr;
            int kb = kGeneral ? f.kv_first : 0;   // key block of stream block j
            if (sparse) kb = sparse_next(f.mrow0, f.mrow1, kb, f.kb_end, lane);
            for (int j = 0; j < f.n_kv && ok; ++j) {
                // K and V of a block complete on the K slot's barrier (one wait for both)
                const uint32_t slot_k = kv_cnt % S;
                for (int kv = 0; kv < 2; ++kv) {
                    const uint32_t slot = kv_cnt % S, ph = (kv_cnt / S) & 1u;
                    ok = warp_wait(bar(Lay::kKVEmpty + slot), ph ^ 1u, w, lane);
                    if (!ok) break;
                    if (lane == 0) {
                        if (kv == 0) mbar_expect_tx(bar(Lay::kKVFull + slot_k), 2 * Lay::kTileBytes);
                        for (int hf = 0; hf < Lay::kHalves; ++hf)
                            tma_load_3d(base + Lay::kKVOff + slot * Lay::kTileBytes + hf * kBox,
                                        kv ? &tmV : &tmK, bar(Lay::kKVFull + slot_k), hf * 64, f.hk,
                                        f.k_row0 + (kGeneral ? kb : j) * kBN);
                    }
                    __syncwarp();
                    ++kv_cnt;
                }
                if constexpr (kGeneral) kb = sparse ? sparse_next(f.mrow0, f.mrow1, kb + 1, f.kb_end, lane) : kb + 1;
            }
            ++it;
        }
        if (lane == 0) {   // let issued copies land before the CTA can exit
            if (q_issued) drain_wait(bar(Lay::kQFull), (q_issued - 1) & 1u, p.wait_budget_ns);
            for (uint32_t i = 0; i < (uint32_t)S && i < kv_cnt; ++i) {
                const uint32_t n = kv_cnt - 1 - i;
                if ((n & 1u) == 0) drain_wait(bar(Lay::kKVFull + n % S), (n / S) & 1u, p.wait_budget_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        setmaxnreg_dec<kRegsLoadMma>();
        constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
        constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, HD, false, true);
        // Descriptors are built once; each MMA adds a compile-time offset to the low half.
        const SmemDesc q_desc[2] = {sdesc_sw128_split(base + Lay::kQOff, 16, 1024),
                                    sdesc_sw128_split(base + Lay::kQOff + Lay::kTileBytes, 16, 1024)};
        const SmemDesc k_desc0 = sdesc_sw128_split(base + Lay::kKVOff, 16, 1024);     // K-major
        const SmemDesc v_desc0 = sdesc_sw128_split(base + Lay::kKVOff, kBox, 1024);   // MN-major
        // S_tq = Q_tq K^T: both operands K-major; 16-column K steps inside a 64-column box.
        auto issue_s = [&](int tq, uint32_t slot) {
            const SmemDesc qd = q_desc[tq];
            SmemDesc kd = k_desc0;
            kd.lo += slot * desc_step(Lay::kTileBytes);
            const uint32_t d_tmem = tmem + (tq ? 128u : 0u);
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t off = desc_step((k >> 2) * kBox + (k & 3) * 32);
                mma_ss(d_tmem, qd, off, kd, off, kIdescS, k > 0);
            }
        };
        // O_tq (+)= P_tq V: P (bf16, 2 per column) from tensor memory, V MN-major in shared memory.
        auto issue_pv = [&](int tq, uint32_t slot, bool acc) {
            SmemDesc vd = v_desc0;
            vd.lo += slot * desc_step(Lay::kTileBytes);
            const uint32_t d_tmem = tmem + (tq ? Lay::kTmemO1 : Lay::kTmemO0);
            const uint32_t p_tmem = tmem + (tq ? Lay::kTmemP1 : Lay::kTmemP0);
#pragma unroll
            for (int k = 0; k < kBN / 16; ++k)
                mma_ts(d_tmem, p_tmem + k * 8, vd, desc_step(k * 2048), kIdescPV, (acc || k > 0) ? 1u : 0u);
        };
        auto issue_s_w = [&](int tq, uint32_t slot) {
            const SmemDesc qd = q_desc[tq];
            SmemDesc kd = k_desc0;
            kd.lo += slot * desc_step(Lay::kTileBytes);
            const uint32_t d_tmem = tmem + (tq ? 128u : 0u);
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t off = desc_step((k >> 2) * kBox + (k & 3) * 32);
                mma_ss_w(d_tmem, qd, off, kd, off, kIdescS, k > 0);
            }
        };
        auto issue_pv_w = [&](int tq, uint32_t slot, bool acc) {
            SmemDesc vd = v_desc0;
            vd.lo += slot * desc_step(Lay::kTileBytes);
            const uint32_t d_tmem = tmem + (tq ? Lay::kTmemO1 : Lay::kTmemO0);
            const uint32_t p_tmem = tmem + (tq ? Lay::kTmemP1 : Lay::kTmemP0);
#pragma unroll
            for (int k = 0; k < kBN / 16; ++k)
                mma_ts_w(d_tmem, p_tmem + k * 8, vd, desc_step(k * 2048), kIdescPV, (acc || k > 0) ? 1u : 0u);
        };
        uint32_t kv_cnt = 0, it = 0, pc0 = 0, pc1 = 0, sf0 = 0, sf1 = 0;
        bool ok = true;
        if constexpr (Lay::kSepP) {
            // Per stream block j: S(j+1) of each Q tile as soon as its softmax has read
            // S(j), then PV(j) of each once its P is written. The next S no longer waits
            // for the current PV, so a Q tile's round trip is its softmax alone. The
            // whole warp runs the issue code and one elected lane issues each MMA: from a
            // one-lane branch the issue rate falls behind the softmax warps sharing its
            // scheduler (this order measured 6-8% slower than the d = 128 order that way,
            // 18-21% faster converged); commits stay on lane 0.
            for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
                const FwdTile f = fwd_tile<kGeneral, kSparse>(t, p, vm, varlen, lane);
                if (f.n_kv == 0) continue;
                const int n0 = f.n_kv0, s1 = kGeneral ? f.kv_start1 : 0;   // Q tile 0: [0, n0), Q tile 1: [s1, n_kv)
                ok = warp_wait(bar(Lay::kQFull), it & 1u, w, lane);
                if (!ok) break;
                uint32_t slot_k = kv_cnt % S;
                ok = warp_wait(bar(Lay::kKVFull + slot_k), (kv_cnt / S) & 1u, w, lane);
                if (!ok) break;
                ++kv_cnt;
                tc_fence_after_sync();
                {
                    if (n0 > 0) {
                        issue_s_w(0, slot_k);
                        if (lane == 0) tc_commit(bar(Lay::kSFull + 0));
                    }
                    if (s1 == 0) {
                        issue_s_w(1, slot_k);
                        if (lane == 0) tc_commit(bar(Lay::kSFull + 1));
                    }
                    if (lane == 0) tc_commit(bar(Lay::kKVEmpty + slot_k));
                    if (f.n_kv == 1) if (lane == 0) tc_commit(bar(Lay::kQEmpty));   // Q is no longer read: the next tile's may land
                }
                __syncwarp();
                for (int j = 0; j < f.n_kv; ++j) {
                    const uint32_t slot_v = kv_cnt % S;   // arrived with the block's K
                    ++kv_cnt;
                    if (j + 1 < f.n_kv) {   // S of block j+1 (K and V of block j+1 land together)
                        slot_k = kv_cnt % S;
                        ok = warp_wait(bar(Lay::kKVFull + slot_k), (kv_cnt / S) & 1u, w, lane);
                        if (!ok) break;
                        ++kv_cnt;
                        if (j + 1 < n0) {   // Q tile 0 saw block j too: its softmax must have read S0(j)
                            ok = warp_wait(bar(Lay::kSFree + 0), sf0 & 1u, w, lane);
                            if (!ok) break;
                            ++sf0;
                            tc_fence_after_sync();
                            {
                                issue_s_w(0, slot_k);
                                if (lane == 0) tc_commit(bar(Lay::kSFull + 0));
                            }
                            __syncwarp();
                        }
                        if (j + 1 >= s1) {
                            if (j >= s1) {   // Q tile 1 saw block j: its softmax must have read S1(j)
                                ok = warp_wait(bar(Lay::kSFree + 1), sf1 & 1u, w, lane);
                                if (!ok) break;
                                ++sf1;
                            }
                            tc_fence_after_sync();
                            {
                                issue_s_w(1, slot_k);
                                if (lane == 0) tc_commit(bar(Lay::kSFull + 1));
                            }
                            __syncwarp();
                        }
                        {
                            if (lane == 0) tc_commit(bar(Lay::kKVEmpty + slot_k));
                            if (j + 2 == f.n_kv) if (lane == 0) tc_commit(bar(Lay::kQEmpty));   // the tile's last S
                        }
                        __syncwarp();
                    }
                    if (j < n0) {   // O0 += P0 V(j)
                        ok = warp_wait(bar(Lay::kPFull + 0), pc0 & 1u, w, lane);
                        if (!ok) break;
                        ++pc0;
                        tc_fence_after_sync();
                        {
                            issue_pv_w(0, slot_v, j > 0);
                            if (lane == 0) tc_commit(bar(j + 1 == n0 ? Lay::kOFull + 0 : Lay::kPVDone + 0));
                        }
                        __syncwarp();
                    }
                    if (j >= s1) {   // O1 += P1 V(j)
                        ok = warp_wait(bar(Lay::kPFull + 1), pc1 & 1u, w, lane);
                        if (!ok) break;
                        ++pc1;
                        tc_fence_after_sync();
                        {
                            issue_pv_w(1, slot_v, j > s1);
                            if (lane == 0) tc_commit(bar(j + 1 == f.n_kv ? Lay::kOFull + 1 : Lay::kPVDone + 1));
                        }
                        __syncwarp();
                    }
                    if (lane == 0) if (lane == 0) tc_commit(bar(Lay::kKVEmpty + slot_v));
                    __syncwarp();
                }
                if (!ok) break;
                ++it;
            }
        } else {
        uint32_t kv_cnt = 0, it = 0, pc0 = 0, pc1 = 0;
        bool ok = true;
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const FwdTile f = fwd_tile<kGeneral, kSparse>(t, p, vm, varlen, lane);
            if (f.n_kv == 0) continue;
            const int n0 = f.n_kv0, s1 = kGeneral ? f.kv_start1 : 0;   // Q tile 0: [0, n0), Q tile 1: [s1, n_kv)
            ok = warp_wait(bar(Lay::kQFull), it & 1u, w, lane);
            if (!ok) break;
            uint32_t slot_k = kv_cnt % S;
            ok = warp_wait(bar(Lay::kKVFull + slot_k), (kv_cnt / S) & 1u, w, lane);
            if (!ok) break;
            ++kv_cnt;
            tc_fence_after_sync();
            if (lane == 0) {
                if (n0 > 0) {
                    issue_s(0, slot_k);
                    tc_commit(bar(Lay::kSFull + 0));
                }
                if (s1 == 0) {
                    issue_s(1, slot_k);
                    tc_commit(bar(Lay::kSFull + 1));
                }
                tc_commit(bar(Lay::kKVEmpty + slot_k));
                if (f.n_kv == 1) tc_commit(bar(Lay::kQEmpty));   // Q is no longer read: the next tile's may land
            }
            __syncwarp();
            for (int j = 0; j < f.n_kv; ++j) {
                const uint32_t slot_v = kv_cnt % S;   // arrived with the block's K
                ++kv_cnt;
                const bool more = j + 1 < f.n_kv;
                // tile 0: PV for block j, then S for block j+1 (while it sees them)
                if (j < n0) {
                    ok = warp_wait(bar(Lay::kPFull + 0), pc0 & 1u, w, lane);
                    if (!ok) break;
                    ++pc0;
                    tc_fence_after_sync();
                    if (lane == 0) issue_pv(0, slot_v, j > 0);
                    __syncwarp();
                }
                if (more) {   // K of block j+1, for tile 1 (and tile 0 if it sees it)
                    slot_k = kv_cnt % S;
                    ok = warp_wait(bar(Lay::kKVFull + slot_k), (kv_cnt / S) & 1u, w, lane);
                    if (!ok) break;
                    ++kv_cnt;
                    tc_fence_after_sync();
                }
                if (lane == 0) {
                    if (j + 1 < n0) {
                        issue_s(0, slot_k);
                        tc_commit(bar(Lay::kSFull + 0));
                    } else if (j + 1 == n0) {
                        tc_commit(bar(Lay::kOFull + 0));   // after PV(0, j): tile 0 is done
                    }
                }
                __syncwarp();
                // tile 1 (from stream block s1 on)
                if (j >= s1) {
                    ok = warp_wait(bar(Lay::kPFull + 1), pc1 & 1u, w, lane);
                    if (!ok) break;
                    ++pc1;
                    tc_fence_after_sync();
                }
                if (lane == 0) {
                    if (j >= s1) issue_pv(1, slot_v, j > s1);
                    tc_commit(bar(Lay::kKVEmpty + slot_v));
                    if (more) {
                        if (j + 1 >= s1) {
                            issue_s(1, slot_k);
                            tc_commit(bar(Lay::kSFull + 1));
                        }
                        tc_commit(bar(Lay::kKVEmpty + slot_k));
                        if (j + 2 == f.n_kv) tc_commit(bar(Lay::kQEmpty));   // that was the tile's last S
                    } else {
                        tc_commit(bar(Lay::kOFull + 1));
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
            ++it;
        }
        }
        if (lane == 0) {   // every MMA issued so far must finish before tensor memory is freed
            tc_commit(bar(Lay::kDrain));
            drain_wait(bar(Lay::kDrain), 0, p.wait_budget_ns);
        }
        __syncwarp();
    } else if (warp < 4) {
        setmaxnreg_dec<kRegsLoadMma>();   // idle warps of the load/MMA warpgroup
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        setmaxnreg_inc<kRegsSoftmax>();
        const int tq = (warp - 4) >> 2;
        const int quarter = warp & 3;                 // tensor-memory lane quarter of this warp
        const int row_in_tile = quarter * 32 + lane;
        const uint32_t t_s = tmem_at(tmem, quarter * 32, tq ? 128u : 0u);
        const uint32_t t_o = tmem_at(tmem, quarter * 32, tq ? Lay::kTmemO1 : Lay::kTmemO0);
        const uint32_t t_p = tmem_at(tmem, quarter * 32, tq ? Lay::kTmemP1 : Lay::kTmemP0);   // bf16 P
        const float sl2 = g.scale_log2;
        uint32_t sc = 0, it = 0, pvc = 0;
        bool ok = true;
        uint32_t rr[32];
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const FwdTile f = fwd_tile<kGeneral, kSparse>(t, p, vm, varlen, lane);
            const int r = f.mp * kRowsPerTile + tq * kBM + row_in_tile;   // row inside the sequence
            const bool valid = r < f.lq;
            const long prow = (long)f.q_row0 + tq * kBM + row_in_tile;   // packed row
            __nv_bfloat16* optr = p.o + (prow * g.H + f.h) * HD;
            float* lptr = varlen ? p.lse + (long)f.h * g.Lq + prow
                                 : p.lse + ((long)f.b * g.H + f.h) * g.Lq + r;
            const int jb = kGeneral && tq ? f.kv_start1 : 0, nkv = tq ? f.n_kv : f.n_kv0;   // stream blocks [jb, nkv)
            if (nkv == 0) {
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(optr);
#pragma unroll
                    for (int c = 0; c < HD / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
                    *lptr = -INFINITY;
                }
                continue;
            }
            const MaskBand mb = mask_band(f.lq, f.lk, g.win_left, g.win_right);
            const int col_lo = kGeneral ? band_key_lo(mb, r) : 0, col_limit = band_key_hi(mb, r);   // keys [col_lo, col_limit)
            // block-sparse: this Q tile's mask row (null: its row block is past the mask, no row is stored)
            const bool sparse = kSparse && f.mrow0 != nullptr;
            const unsigned char* mrow = tq ? f.mrow1 : f.mrow0;
            int kb = (kGeneral ? f.kv_first : 0) + jb;   // key block of stream block j
            if (sparse) kb = sparse_next(f.mrow0, f.mrow1, f.kv_first, f.kb_end, lane);
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = jb; j < nkv; ++j) {
                ok = warp_wait(bar(Lay::kSFull + tq), sc & 1u, w, lane);
                if (!ok) break;
                ++sc;
                tc_fence_after_sync();
                float s[kBN];
                {
                    uint32_t r128[kBN];
                    tmem_ld128(t_s, r128);
#pragma unroll
                    for (int i = 0; i < kBN; ++i) s[i] = u2f(r128[i]);
                }
                if constexpr (Lay::kSepP) {   // S is in registers: the MMA warp may compute the next one
                    if (j + 1 < nkv) {
                        tc_fence_before_sync();
                        mbar_arrive(bar(Lay::kSFree + tq));
                    }
                }
                const int c0 = (kGeneral ? kb : j) * kBN;
                const bool dropped = sparse && (mrow == nullptr || mrow[kb] == 0);   // the block mask drops it here
                if (dropped || c0 + kBN > col_limit || c0 < col_lo) {
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (dropped || c0 + c >= col_limit || c0 + c < col_lo) s[c] = -INFINITY;
                }
                if constexpr (kGeneral) kb = sparse ? sparse_next(f.mrow0, f.mrow1, kb + 1, f.kb_end, lane) : kb + 1;
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int c = 4; c < kBN; c += 4) {
                    mx0 = fmaxf(mx0, s[c]);
                    mx1 = fmaxf(mx1, s[c + 1]);
                    mx2 = fmaxf(mx2, s[c + 2]);
                    mx3 = fmaxf(mx3, s[c + 3]);
                }
                const float m_new = fmaxf(m_run, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2);
                const bool need = m_new > m_run + kTau;
                bool pv_seen = !(Lay::kSepP && j > jb);   // (d = 64) PV(j-1) has completed
                if (__any_sync(kFullMask, need)) {
                    const float alpha = (m_new == -INFINITY) ? 1.f : ex2_mufu(m_run - m_new);
                    if (!pv_seen) {
                        ok = warp_wait(bar(Lay::kPVDone + tq), pvc & 1u, w, lane);
                        if (!ok) break;
                        ++pvc;
                        pv_seen = true;
                        tc_fence_after_sync();
                    }
                    if (j > jb) {   // O holds blocks jb..j-1 (their MMAs completed before S_j did, or PV(j-1) did)
#pragma unroll
                        for (int c = 0; c < HD / 32; ++c) {
                            tmem_ld32(t_o + c * 32, rr);
#pragma unroll
                            for (int i = 0; i < 32; ++i) rr[i] = f2u(u2f(rr[i]) * alpha);
                            tmem_st32(t_o + c * 32, rr);
                        }
                    }
                    l_run *= alpha;
                    m_run = m_new;
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                if (!pv_seen) {   // (d = 64) PV(j-1) has read the P buffer this block's P goes to
                    ok = warp_wait(bar(Lay::kPVDone + tq), pvc & 1u, w, lane);
                    if (!ok) break;
                    ++pvc;
                    tc_fence_after_sync();
                }
                float l0 = 0.f, l1 = 0.f;
                if constexpr (kPoly > 0) {
                    if (j + 1 < nkv) exp_row_to_tmem<kPoly>(s, sl2, neg_m, t_p, l0, l1);
                    else exp_row_to_tmem<0>(s, sl2, neg_m, t_p, l0, l1);   // last block: MUFU only
                } else {
                    exp_row_to_tmem<0>(s, sl2, neg_m, t_p, l0, l1);   // one copy of the loop in the code
                }
                l_run += l0 + l1;
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(bar(Lay::kPFull + tq));
            }
            if (!ok) break;
            ok = warp_wait(bar(Lay::kOFull + tq), it & 1u, w, lane);
            if (!ok) break;
            ++it;
            tc_fence_after_sync();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                tmem_ld32(t_o + c * 32, rr);
                if (valid) {
                    uint32_t o2[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        o2[i] = pack_bf16x2(u2f(rr[2 * i]) * inv_l, u2f(rr[2 * i + 1]) * inv_l);
                    uint4* dst = reinterpret_cast<uint4*>(optr + c * 32);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(o2[4 * v4], o2[4 * v4 + 1], o2[4 * v4 + 2], o2[4 * v4 + 3]);
                }
            }
            if (valid) *lptr = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
            tc_fence_before_sync();
        }
    }
    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// The kernel for a problem: the general one for a left window bound or a block
// mask (MUFU only), else the plain one with the requested exp2 emulation.
template <int HD>
auto fwd_kernel_for(const FwdParams& p, int poly_every) {
    if (p.mask.ptr) return fwd_kernel<HD, true, true, 0>;
    if (p.g.win_left >= 0) return fwd_kernel<HD, true, false, 0>;
    return poly_every == 8 ? fwd_kernel<HD, false, false, 8>
                           : (poly_every == 4 ? fwd_kernel<HD, false, false, 4> : fwd_kernel<HD, false, false, 0>);
}

template <int HD>
cudaError_t launch_fwd_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdParams& p, int poly_every, int num_sms, cudaStream_t stream) {
    using Lay = FwdLayout<HD>;
    auto kern = fwd_kernel_for<HD>(p, poly_every);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    // the register split re-distributes exactly the registers the CTA launches with
    if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    const int grid = p.g.cu_seqlens ? num_sms : min(p.n_tiles, num_sms);
    if (grid <= 0) return cudaSuccess;
    kern<<<grid, kThreads, Lay::kSmemBytes, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int poly_every, int num_sms, cudaStream_t stream) {
    switch (p.g.d) {
        case 64: return launch_fwd_hd<64>(tq, tk, tv, p, poly_every, num_sms, stream);
        case 128: return launch_fwd_hd<128>(tq, tk, tv, p, poly_every, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
