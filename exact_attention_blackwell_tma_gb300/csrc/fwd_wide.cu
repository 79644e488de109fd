// Forward kernel for head dims above 128: d = 192, 256, and d_qk = 192 with
// d_v = 128 (the FlashAttention-4 paper's Section 5.1, Fig. 5 shape).
//
// Same operation and warp roles as fwd.cu, but tensor memory cannot hold two
// Q tiles' S and O at these head dims (2 x (128 + d) > 512 columns), so a work
// tile is ONE 128-row Q tile and the overlap of MMA and softmax comes from a
// double-buffered S instead of the ping-pong of two Q tiles (FlashAttention-4
// paper, Section 3.1.2, describes the tensor-memory budget that forces this
// trade at large head dims):
//  * tensor memory: S buffers at columns 0 and 128 (fp32, P written as bf16
//    over the first 64 columns of its buffer), O at 256 (d columns);
//  * MMA order: S(0), S(1), then for each block j: PV(j) once P(j) is ready,
//    then S(j+2) into the buffer P(j) occupied (the tensor pipe executes in
//    issue order, so PV(j) has read P(j) before S(j+2) overwrites it);
//  * while the softmax works on S(j+1), PV(j) may still be running, so a
//    rescale of O first waits for PV(j-1) to complete (rare: the running max
//    moves only when it grows by more than kTau);
//  * K/V tiles are loaded in consumption order K0, K1, V0, K2, V1, K3, ...
// Every wait is bounded, as in fwd.cu.
#include "kernels.h"
#include "ptx.cuh"
#include "mask.cuh"
#include "sched.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 256;       // 8 warps: load, MMA, 2 idle, 4 softmax
constexpr float kTau = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 16384;

// HD: head dim of q and k; DV: head dim of v and O (equal except for the
// d_qk = 192, d_v = 128 shape).
template <int HD, int DV>
struct WideLayout {
    static constexpr int kHalves = HD / 64;               // 64-column boxes of a Q/K row
    static constexpr int kHalvesV = DV / 64;              // ... of a V row
    static constexpr int kTileBytes = kBM * HD * 2;       // Q/K tile; ring slots have this size
    static constexpr int kStages = HD == 192 ? 3 : 2;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = kTileBytes;
    static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
    // S and P barriers come one per S buffer: a single P barrier could complete
    // twice (P of blocks j and j+1) before the MMA warp waits on it.
    static constexpr int kQFull = 0, kQEmpty = 1, kKVFull = 2, kKVEmpty = 2 + kStages, kSFull = 2 + 2 * kStages,
                         kPFull = kSFull + 2, kPVDone = kPFull + 2, kOFull = kPVDone + 1, kDrain = kOFull + 1,
                         kNumBars = kDrain + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kMapOff = (kMiscOff + 16 + 15) / 16 * 16;
    static constexpr int kSmemBytes = kMapOff + (int)sizeof(VarlenMap) + 1024;
    static constexpr uint32_t kTmemO = 256;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(256 + DV <= (int)kTmemCols, "tensor memory budget");
    static_assert(DV <= HD, "a V tile must fit a ring slot");
};

struct WideTile {
    int b, h, m;     // batch, query head, 128-row query block
    int hk;          // key/value head read by query head h
    int lq, lk;
    int q_row0;      // packed row of the tile's first query row
    int k_row0;
    int kv_first, n_kv;   // K/V blocks kv_first .. kv_first + n_kv - 1 (n_kv = 0: no row sees a key)
    // block-sparse (block mask given): the n_kv blocks in [kv_first, kb_end)
    // that the tile's mask row keeps
    const unsigned char* mrow;
    int kb_end;
};

// kSparse: a block mask may be given (the kernels without one contain no mask scans)
template <bool kSparse>
__device__ __forceinline__ WideTile wide_tile(int t, const FwdParams& p, const VarlenMap& vm, bool varlen, int lane) {
    const Geometry& g = p.g;
    Tile ti = varlen ? sched_varlen(vm, t, g.B, g.H, kBM, p.head_section, g.causal != 0, false)
                     : (g.causal ? sched_dense_lpt(t, g.B, g.H, p.nm, true)
                                 : sched_dense(t, g.H, p.nm, p.head_section, false));
    WideTile f;
    f.b = ti.b;
    f.h = ti.h;
    f.hk = ti.h / g.group;
    f.m = ti.m;
    if (varlen) {
        f.lq = vm_lq(vm, ti.b);
        f.lk = vm_lk(vm, ti.b);
        f.q_row0 = vm.start[ti.b] + ti.m * kBM;
        f.k_row0 = vm.start_k[ti.b];
    } else {
        f.lq = g.Lq;
        f.lk = g.Lk;
        f.q_row0 = ti.b * g.Lq + ti.m * kBM;
        f.k_row0 = ti.b * g.Lk;
    }
    const MaskBand mb = mask_band(f.lq, f.lk, g.win_left, g.win_right);
    int jlo, jhi;
    band_key_blocks(mb, ti.m * kBM, ti.m * kBM + kBM - 1, kBN, &jlo, &jhi);
    f.kv_first = jlo;
    f.n_kv = jhi - jlo;
    f.kb_end = jhi;
    f.mrow = nullptr;
    if constexpr (kSparse) {
        if (p.mask.ptr) {
            const int mh = p.mask.heads == 1 ? 0 : ti.h;
            f.mrow = p.mask.ptr + ((long)mh * mask_rows(g) + ti.m) * mask_cols(g);
            f.n_kv = f.n_kv > 0 ? sparse_count(f.mrow, nullptr, jlo, jhi, lane) : 0;
        }
    }
    return f;
}

template <int HD, int DV, bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
fwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using Lay = WideLayout<HD, DV>;
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
        mbar_init(bar(Lay::kSFull + 0), 1);
        mbar_init(bar(Lay::kSFull + 1), 1);
        mbar_init(bar(Lay::kPFull + 0), 128);
        mbar_init(bar(Lay::kPFull + 1), 128);
        mbar_init(bar(Lay::kPVDone), 1);
        mbar_init(bar(Lay::kOFull), 1);
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
        sched_varlen_build(vm, g.cu_seqlens, g.cu_seqlens_k, g.B, g.H, kBM, false, tid, kThreads);
        n_tiles = vm.pre[g.B];
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{abort_flag, p.status, p.wait_budget_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        uint32_t kv_cnt = 0, it = 0, q_issued = 0;
        bool ok = true;
        // one tile of K (kv = 0) or V (kv = 1) of key block kb, into the next ring slot
        auto load_kv = [&](const WideTile& f, int kv, int kb) -> bool {
            const uint32_t slot = kv_cnt % S, ph = (kv_cnt / S) & 1u;
            if (!warp_wait(bar(Lay::kKVEmpty + slot), ph ^ 1u, w, lane)) return false;
            if (lane == 0) {
                const int boxes = kv ? Lay::kHalvesV : Lay::kHalves;
                mbar_expect_tx(bar(Lay::kKVFull + slot), boxes * kBox);
                for (int hf = 0; hf < boxes; ++hf)
                    tma_load_3d(base + Lay::kKVOff + slot * Lay::kTileBytes + hf * kBox, kv ? &tmV : &tmK,
                                bar(Lay::kKVFull + slot), hf * 64, f.hk, f.k_row0 + kb * kBN);
            }
            __syncwarp();
            ++kv_cnt;
            return true;
        };
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const WideTile f = wide_tile<kSparse>(t, p, vm, varlen, lane);
            if (f.n_kv == 0) continue;
            ok = warp_wait(bar(Lay::kQEmpty), (it & 1u) ^ 1u, w, lane);
            if (!ok) break;
            if (lane == 0) {
                mbar_expect_tx(bar(Lay::kQFull), Lay::kTileBytes);
                for (int hf = 0; hf < Lay::kHalves; ++hf)
                    tma_load_3d(base + Lay::kQOff + hf * kBox, &tmQ, bar(Lay::kQFull), hf * 64, f.h, f.q_row0);
            }
            __syncwarp();
            ++q_issued;
            // consumption order: K0, K1, then V_j, K_{j+2} for each block j; the K and
            // V cursors walk the tile's key blocks (block-sparse: the kept ones)
            const bool sparse = kSparse && f.mrow != nullptr;
            auto kept = [&](int kb) { return sparse ? sparse_next(f.mrow, nullptr, kb, f.kb_end, lane) : kb; };
            int kb_k = kept(f.kv_first), kb_v = kb_k;
            ok = load_kv(f, 0, kb_k);
            kb_k = kept(kb_k + 1);
            if (ok && f.n_kv >= 2) {
                ok = load_kv(f, 0, kb_k);
                kb_k = kept(kb_k + 1);
            }
            for (int j = 0; j < f.n_kv && ok; ++j) {
                ok = load_kv(f, 1, kb_v);
                kb_v = kept(kb_v + 1);
                if (ok && j + 2 < f.n_kv) {
                    ok = load_kv(f, 0, kb_k);
                    kb_k = kept(kb_k + 1);
                }
            }
            ++it;
        }
        if (lane == 0) {
            if (q_issued) drain_wait(bar(Lay::kQFull), (q_issued - 1) & 1u, p.wait_budget_ns);
            for (uint32_t i = 0; i < (uint32_t)S && i < kv_cnt; ++i) {
                const uint32_t n = kv_cnt - 1 - i;
                drain_wait(bar(Lay::kKVFull + n % S), (n / S) & 1u, p.wait_budget_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
        constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, DV, false, true);
        const SmemDesc q_desc = sdesc_sw128_split(base + Lay::kQOff, 16, 1024);
        const SmemDesc k_desc0 = sdesc_sw128_split(base + Lay::kKVOff, 16, 1024);
        const SmemDesc v_desc0 = sdesc_sw128_split(base + Lay::kKVOff, kBox, 1024);
        uint32_t kv_cnt = 0, it = 0, pc[2] = {0, 0};
        bool ok = true;
        // wait for the next ring slot in consumption order; returns the slot
        auto next_slot = [&](uint32_t& slot) -> bool {
            slot = kv_cnt % S;
            if (!warp_wait(bar(Lay::kKVFull + slot), (kv_cnt / S) & 1u, w, lane)) return false;
            ++kv_cnt;
            tc_fence_after_sync();
            return true;
        };
        auto issue_s = [&](uint32_t buf, uint32_t slot) {
            SmemDesc kd = k_desc0;
            kd.lo += slot * desc_step(Lay::kTileBytes);
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t off = desc_step((k >> 2) * kBox + (k & 3) * 32);
                mma_ss(tmem + 128u * buf, q_desc, off, kd, off, kIdescS, k > 0);
            }
            tc_commit(bar(Lay::kSFull + buf));
            tc_commit(bar(Lay::kKVEmpty + slot));
        };
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const WideTile f = wide_tile<kSparse>(t, p, vm, varlen, lane);
            if (f.n_kv == 0) continue;
            ok = warp_wait(bar(Lay::kQFull), it & 1u, w, lane);
            if (!ok) break;
            uint32_t slot;
            ok = next_slot(slot);
            if (!ok) break;
            if (lane == 0) {
                issue_s(0, slot);
                if (f.n_kv == 1) tc_commit(bar(Lay::kQEmpty));
            }
            __syncwarp();
            if (f.n_kv > 1) {
                ok = next_slot(slot);
                if (!ok) break;
                if (lane == 0) {
                    issue_s(1, slot);
                    if (f.n_kv == 2) tc_commit(bar(Lay::kQEmpty));
                }
                __syncwarp();
            }
            for (int j = 0; j < f.n_kv; ++j) {
                uint32_t slot_v;
                ok = next_slot(slot_v);
                if (!ok) break;
                ok = warp_wait(bar(Lay::kPFull + (j & 1)), pc[j & 1] & 1u, w, lane);
                if (!ok) break;
                ++pc[j & 1];
                tc_fence_after_sync();
                if (lane == 0) {
                    SmemDesc vd = v_desc0;
                    vd.lo += slot_v * desc_step(Lay::kTileBytes);
                    const uint32_t p_tmem = tmem + 128u * (uint32_t)(j & 1);
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        mma_ts(tmem + Lay::kTmemO, p_tmem + kk * 8, vd, desc_step(kk * 2048), kIdescPV,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar(Lay::kPVDone));
                    tc_commit(bar(Lay::kKVEmpty + slot_v));
                    if (j + 1 == f.n_kv) tc_commit(bar(Lay::kOFull));
                }
                __syncwarp();
                if (j + 2 < f.n_kv) {
                    uint32_t slot_k;
                    ok = next_slot(slot_k);
                    if (!ok) break;
                    if (lane == 0) {
                        issue_s((uint32_t)(j & 1), slot_k);
                        if (j + 3 == f.n_kv) tc_commit(bar(Lay::kQEmpty));   // the tile's last S
                    }
                    __syncwarp();
                }
            }
            if (!ok) break;
            ++it;
        }
        if (lane == 0) {
            tc_commit(bar(Lay::kDrain));
            drain_wait(bar(Lay::kDrain), 0, p.wait_budget_ns);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax warpgroup
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_o = tmem + lane_off + Lay::kTmemO;
        const float sl2 = g.scale_log2;
        uint32_t sc[2] = {0, 0}, it = 0, pv_seen = 0;
        bool ok = true;
        uint32_t rr[32];
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const WideTile f = wide_tile<kSparse>(t, p, vm, varlen, lane);
            const int r = f.m * kBM + row_in_tile;
            const bool valid = r < f.lq;
            const long prow = (long)f.q_row0 + row_in_tile;
            __nv_bfloat16* optr = p.o + (prow * g.H + f.h) * DV;
            float* lptr = varlen ? p.lse + (long)f.h * g.Lq + prow : p.lse + ((long)f.b * g.H + f.h) * g.Lq + r;
            if (f.n_kv == 0) {
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(optr);
#pragma unroll
                    for (int c = 0; c < DV / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
                    *lptr = -INFINITY;
                }
                continue;
            }
            const MaskBand mb = mask_band(f.lq, f.lk, g.win_left, g.win_right);
            const int col_lo = band_key_lo(mb, r), col_limit = band_key_hi(mb, r);   // keys [col_lo, col_limit)
            const bool sparse = kSparse && f.mrow != nullptr;
            int kb = sparse ? sparse_next(f.mrow, nullptr, f.kv_first, f.kb_end, lane) : f.kv_first;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < f.n_kv; ++j) {
                const int buf = j & 1;
                ok = warp_wait(bar(Lay::kSFull + buf), sc[buf] & 1u, w, lane);
                if (!ok) break;
                ++sc[buf];
                tc_fence_after_sync();
                const uint32_t t_s = tmem + lane_off + 128u * (uint32_t)buf;
                float s[kBN];
                {
                    uint32_t r128[kBN];
                    tmem_ld128(t_s, r128);
#pragma unroll
                    for (int i = 0; i < kBN; ++i) s[i] = u2f(r128[i]);
                }
                const int c0 = kb * kBN;
                kb = sparse ? sparse_next(f.mrow, nullptr, kb + 1, f.kb_end, lane) : kb + 1;
                if (c0 + kBN > col_limit || c0 < col_lo) {
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (c0 + c >= col_limit || c0 + c < col_lo) s[c] = -INFINITY;
                }
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
                if (__any_sync(kFullMask, need)) {
                    const float alpha = (m_new == -INFINITY) ? 1.f : ex2_mufu(m_run - m_new);
                    if (j > 0) {
                        // O must hold blocks 0..j-1: wait for PV(j-1), the (pv_seen + j)-th PV overall
                        ok = warp_wait(bar(Lay::kPVDone), (pv_seen + j - 1) & 1u, w, lane);
                        if (!ok) break;
                        tc_fence_after_sync();
#pragma unroll
                        for (int c = 0; c < DV / 32; ++c) {
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
                // x = s * sl2 - m and the row sum on packed fp32 pairs
                const uint64_t sc2 = f32x2(sl2, sl2), nm2 = f32x2(neg_m, neg_m);
                uint64_t acc_a = f32x2(0.f, 0.f), acc_b = acc_a;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float x0, x1;
                        f32x2_split(ffma2(f32x2(s[64 * hf + 2 * i], s[64 * hf + 2 * i + 1]), sc2, nm2), x0, x1);
                        const float p0 = ex2_mufu(x0), p1 = ex2_mufu(x1);
                        if (i & 1) acc_b = fadd2(acc_b, f32x2(p0, p1));
                        else acc_a = fadd2(acc_a, f32x2(p0, p1));
                        rr[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(t_s + 32 * hf, rr);
                }
                float l0, l1;
                f32x2_split(fadd2(acc_a, acc_b), l0, l1);
                l_run += l0 + l1;
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(bar(Lay::kPFull + buf));
            }
            if (!ok) break;
            pv_seen += f.n_kv;
            ok = warp_wait(bar(Lay::kOFull), it & 1u, w, lane);
            if (!ok) break;
            ++it;
            tc_fence_after_sync();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c = 0; c < DV / 32; ++c) {
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
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int HD, int DV>
cudaError_t launch_fwd_wide_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const FwdParams& p, int num_sms, cudaStream_t stream) {
    using Lay = WideLayout<HD, DV>;
    auto kern = p.mask.ptr ? fwd_wide_kernel<HD, DV, true> : fwd_wide_kernel<HD, DV, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = p.g.cu_seqlens ? num_sms : min(p.n_tiles, num_sms);
    if (grid <= 0) return cudaSuccess;
    kern<<<grid, kThreads, Lay::kSmemBytes, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, int num_sms, cudaStream_t stream) {
    if (p.g.d == 192 && p.dv == 192) return launch_fwd_wide_hd<192, 192>(tq, tk, tv, p, num_sms, stream);
    if (p.g.d == 256 && p.dv == 256) return launch_fwd_wide_hd<256, 256>(tq, tk, tv, p, num_sms, stream);
    if (p.g.d == 192 && p.dv == 128) return launch_fwd_wide_hd<192, 128>(tq, tk, tv, p, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
