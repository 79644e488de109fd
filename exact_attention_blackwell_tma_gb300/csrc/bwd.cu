// Backward pass: dQ, dK, dV of L = sum(O * dO).
//
// FlashAttention-4 paper, Section 3.2.2: the backward pass runs five MMAs --
// S recomputed, dP = dO V^T, dV += P^T dO, dK += dS^T Q, dQ += dS K -- and
// iterates along the K/V sequence dimension, computing transposed tiles
// (S^T, P^T, dP^T, dS^T) so that the dV product can read P^T from tensor
// memory; dQ is accumulated with global atomics. Tensor memory holds four
// 128-column blocks: S^T (P^T written over it), dP^T (dS^T and the dQ tile
// reuse it), dV and dK; at d = 64 the dQ tile and dS^T have columns of their
// own, and the next query block's dP^T is issued ahead of dK and dQ (B2 H16
// L8192 d64 causal 559 -> 668 TF/s, deterministic 316 -> 466). Section 3.2.4:
// a deterministic mode serialises every dQ tile's accumulation behind a
// semaphore in a fixed order.
//
// Kernels (all on the caller's stream):
//   bwd_prep     D_i = <dO_i, O_i> (fp32), zero the fp32 dQ accumulator and the
//                semaphores, build the longest-first varlen map;
//   bwd_kernel   persistent, one work tile = one 128-key block of one
//                (batch, head); warp 0 TMA, warp 1 MMA, warps 4-11 two compute
//                warpgroups (query columns 0-63 / 64-127 of each tile, one key
//                row per thread), warps 12-15 read dQ tiles out of tensor
//                memory and add them to the fp32 accumulator;
//   bwd_convert  dQ = scale * accumulator -> bf16.
#include "kernels.h"
#include "ptx.cuh"
#include "mask.cuh"
#include "sched.cuh"
#include "dq_order.cuh"
#include "dq_reduce.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;              // query rows per Q block
constexpr int kBN = 128;              // keys per K/V block (work tile)
constexpr int kThreads = 512;         // 16 warps
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 16384;           // 128 rows x 64 bf16 columns
// Register split: 512 threads launch with 128 registers each; the load/MMA
// warpgroup gives 56 up and the dQ warpgroup (which holds a whole 128-column
// dQ row) takes them; the compute warpgroups keep their 128.
constexpr int kLaunchRegs = 128;
constexpr uint32_t kRegsLoadMma = 72, kRegsCompute = 128, kRegsDq = 184;
static_assert((kRegsLoadMma + 2 * kRegsCompute + kRegsDq) * 128 <= kLaunchRegs * kThreads, "register split");

// TMEM column of the bf16 operand (P^T or dS^T) for the k-th 16-query step:
// queries [64 wg, 64 wg + 64) sit in the first 32 columns of the block at 64 wg.
__device__ __forceinline__ uint32_t packed_col(int k) { return (uint32_t)((k >> 2) * 64 + (k & 3) * 8); }
// ... of dS^T in its own 64-column block (d = 64): warpgroup wg's queries in columns [32 wg, 32 wg + 32).
__device__ __forceinline__ uint32_t packed_col_ds(int k) { return (uint32_t)((k >> 2) * 32 + (k & 3) * 8); }

template <int HD>
struct BwdLayout {
    static constexpr int kHalves = HD / 64;
    static constexpr int kTileBytes = kBM * HD * 2;
    // Q and dO have rings of their own: dO is consumed by dP^T and dV early in a
    // query block, Q only by dK at its end, so one dO buffer suffices at d = 128.
    // The space saved holds a second dS tile, so the next dS can be written while
    // the previous dQ tile is still being staged through the other one.
    static constexpr int kQStages = HD == 64 ? 3 : 2;
    static constexpr int kDOStages = HD == 64 ? 2 : 1;
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kTileBytes;
    static constexpr int kQOff = 2 * kTileBytes;                     // Q ring
    static constexpr int kDOOff = kQOff + kQStages * kTileBytes;     // dO ring
    static constexpr int kDSOff = kDOOff + kDOStages * kTileBytes;   // two dS^T tiles, 128 x 128 bf16 each
    static constexpr int kDSBytes = 2 * kBox;
    static constexpr int kStatOff = kDSOff + 2 * kDSBytes;           // per Q stage: -lse2[128], -D[128]
    static constexpr int kBarOff = kStatOff + kQStages * 1024;
    static constexpr int kKVFull = 0, kKVEmpty = 1, kQFull = 2, kQEmpty = kQFull + kQStages,
                         kDOFull = kQEmpty + kQStages, kDOEmpty = kDOFull + kDOStages,
                         kSFull = kDOEmpty + kDOStages, kDPFull = kSFull + 1,
                         kPFull = kDPFull + 1, kDSFull = kPFull + 1, kDSEmpty = kDSFull + 1,   // two
                         kDQFull = kDSEmpty + 2, kDQFree = kDQFull + 1, kDKVFull = kDQFree + 1,
                         kSemGo = kDKVFull + 1, kRedDone = kSemGo + 1, kDrain = kRedDone + 1,
                         kTDSFree = kDrain + 1, kNumBars = kTDSFree + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16;
    // tensor memory columns. Compute warpgroup wg owns query columns
    // [64 wg, 64 wg + 64) of the S^T and dP^T blocks and writes its bf16 P^T and
    // dS^T (two per column) into the first 32 columns of that range, so neither
    // warpgroup ever overwrites a column the other has yet to read.
    static constexpr uint32_t kTS = 0, kTDP = 128, kTDV = 256, kTDK = 256 + HD;
    // d = 64 leaves 128 columns free: the dQ tile and the bf16 dS^T get columns
    // of their own (dQ at 384, dS^T at 448, 32 per warpgroup), so dP^T of the
    // next query block no longer waits for the dQ tile to leave tensor memory
    // nor for dK to read dS^T (kSplitDP). At d = 128 both live in the dP^T block.
    static constexpr bool kSplitDP = HD == 64;
    static constexpr uint32_t kTDQ = kSplitDP ? 384 : kTDP, kTDS = kSplitDP ? 448 : kTDP;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(256 + 2 * HD + (kSplitDP ? 128 : 0) <= (int)kTmemCols, "tensor memory budget");
};

struct BwdTile {
    int b, h, n;       // batch, key/value head, 128-key block
    int lq, lk;
    int q_row0;        // packed row of query 0 of the sequence
    int k_row0;        // packed row of key 0 of the sequence
    int m_begin, m_end;  // 128-row query blocks that see this key block
    int hq0;           // first query head the tile visits
    int nblk;          // query blocks the tile visits: (group / split) x (m_end - m_begin)
    int s;             // which of the key block's split tiles (0 when split == 1)
    // block-sparse (block mask given): entry (query head h, query block m) of
    // this key block's mask column is mcol[h * mhead + m * mstride] (mhead 0:
    // one mask for all heads); nblk counts the kept pairs only
    const unsigned char* mcol;
    long mstride, mhead;
    int nheads;          // query heads the tile visits
};

// The tile's query blocks in visiting order: every query head of its share of
// the group (the whole group unless split, so dK and dV of the block collect
// it in tensor memory), each over [m_begin, m_end). kGQA = false (one query
// head per key/value head): the head never changes.
struct QWalk {
    int h, m;   // query head, 128-row query block
    template <bool kGQA>
    __device__ __forceinline__ void next(const BwdTile& f) {
        ++m;
        if (kGQA && m == f.m_end) {
            m = f.m_begin;
            ++h;
        }
    }
};
__device__ __forceinline__ QWalk qwalk(const BwdTile& f) { return QWalk{f.hq0, f.m_begin}; }

// Block-sparse walk: from (qw.h, qw.m) on, the first pair the block mask keeps
// (warp-wide scans: every lane of the warp calls it alike).
__device__ __forceinline__ void sparse_seek(const BwdTile& f, QWalk& qw, int lane) {
    while (qw.h < f.hq0 + f.nheads) {
        qw.m = sparse_next_col(f.mcol + qw.h * f.mhead, f.mstride, qw.m, f.m_end, lane);
        if (qw.m < f.m_end) return;
        ++qw.h;
        qw.m = f.m_begin;
    }
}

// The first pair of the tile's walk, and the next one.
template <bool kSparse>
__device__ __forceinline__ QWalk qwalk_start(const BwdTile& f, int lane) {
    QWalk qw = qwalk(f);
    if (kSparse && f.mcol) sparse_seek(f, qw, lane);
    return qw;
}
template <bool kGQA, bool kSparse>
__device__ __forceinline__ void qwalk_step(QWalk& qw, const BwdTile& f, int lane) {
    if (kSparse && f.mcol) {
        ++qw.m;
        sparse_seek(f, qw, lane);
    } else {
        qw.next<kGQA>(f);
    }
}


__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// kGQA: grouped heads (the kernels for one query head per key/value head are
// instantiated without the group walk and the split, which keeps their code
// and registers as small as before grouped heads existed)
// kSpt (the deterministic kernels): with a right mask bound, key blocks are
// walked shortest first -- the last key block of a (batch, head) first -- so
// that, with each dQ tile's contributions serialised from its highest key
// block down, no work tile waits at its first dQ write (FlashAttention-4
// paper, Section 3.2.4, SPT order).
template <bool kGQA, bool kBand, bool kSparse, bool kSpt>
__device__ __forceinline__ BwdTile bwd_tile(int t, const BwdParams& p, const VarlenMap* vm, int lane) {
    const Geometry& g = p.g;
    // the split tiles of one key block are neighbours in the walk, so they run
    // at the same time and share the block's K and V in L2
    int sp = 0;
    if constexpr (kGQA) {
        sp = t % p.split;
        t /= p.split;
    }
    // Dense problems walk the heads in L2-sized sections, longest key blocks first
    // within a section (FlashAttention-4 paper, Section 3.3): a section's Q, dO and
    // dQ accumulator stay in L2 (B1 H32 L32768 causal: 43 -> 9.5 GB of DRAM traffic
    // per launch, 975 -> 1045 TF/s). Causal problems whose sections would leave the
    // CTAs unbalanced keep one global longest-first order (p.sections, chosen on
    // the host by sched_sections_pay); the deterministic kernels keep one global
    // order too, shortest first (SPT), which their dQ turns need.
    const bool spt = kSpt && g.causal;
    Tile ti = vm ? sched_varlen(*vm, t, g.B, g.Hkv, kBN, p.head_section, spt, true)
                 : ((g.causal && (spt || !p.sections)) ? sched_dense_lpt(t, g.B, g.Hkv, p.nm, spt)
                                                        : sched_dense(t, g.Hkv, p.nm, p.head_section, false));
    BwdTile f;
    f.b = ti.b;
    f.h = ti.h;
    f.n = ti.m;   // ascending: for causal the smallest key blocks carry the most work
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
        if (g.causal) f.m_begin = max(0, floor_div(f.n * kBN - (f.lk - f.lq), kBM));
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

// ----------------------------------------------------------------------------
// Preprocess: D = rowsum(dO * O), zero the dQ accumulator and semaphores,
// build the varlen map (block 0). D: eight lanes per (row, head), lane l
// reading 16-byte pieces l, l + 8, ... of the row's O and dO (128-byte runs,
// all loads of a lane issued together), summed by shuffles within the eight.
// The loop runs warp by warp, four rows per warp and step, so every shuffle
// has the whole warp.
__global__ void bwd_prep(BwdParams p, VarlenMap* vm_out, long rows_q, long n_acc4, int n_sem, int keys_per_tile) {
    const Geometry& g = p.g;
    const long stride = (long)gridDim.x * blockDim.x;
    const long tid = (long)blockIdx.x * blockDim.x + threadIdx.x;
    const int dv = p.d_v;   // O and dO have the head dim of v: 64 .. 256, 4 pieces of 8 lanes at most
    const int pieces = dv / 64;
    const int lane = threadIdx.x & 31, l8 = lane & 7;
    const long n_rows = rows_q * g.H;
    const long warps = stride / 32;
    for (long r0 = tid / 32 * 4; r0 < n_rows; r0 += warps * 4) {
        const long i = r0 + (lane >> 3);   // (row, head) of this lane's group
        const bool valid = i < n_rows;
        const uint4* o4 = reinterpret_cast<const uint4*>(p.o + (valid ? i : 0) * dv);
        const uint4* d4 = reinterpret_cast<const uint4*>(p.dout + (valid ? i : 0) * dv);
        uint4 a[4], b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (valid && j < pieces) {
                a[j] = o4[j * 8 + l8];
                b[j] = d4[j * 8 + l8];
            }
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (!valid || j >= pieces) continue;
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[j]);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[j]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fa = __bfloat1622float2(a2[e]), fb = __bfloat1622float2(b2[e]);
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (valid && l8 == 0) {
            const long row = i / g.H;
            const int h = (int)(i - row * g.H);
            long di;
            if (g.cu_seqlens) {
                di = (long)h * g.Lq + row;
            } else {
                const long b = row / g.Lq, r = row - b * g.Lq;
                di = (b * g.H + h) * g.Lq + r;
            }
            p.delta[di] = acc;
        }
    }
    float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
    for (long i = tid; i < n_acc4; i += stride) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long i = tid; i < n_sem; i += stride) p.semaphores[i] = 0;
    if (g.cu_seqlens && blockIdx.x == 0) {
        // longest-first map of the sequences (FlashAttention-4 paper, Section 3.3,
        // varlen LPT); work tiles are key blocks (or key-block pairs) of key/value heads
        sched_varlen_build(*vm_out, g.cu_seqlens, g.cu_seqlens_k, g.B, g.Hkv, keys_per_tile, true, threadIdx.x,
                           blockDim.x);
    }
}

// Split grouped heads: dK = scale * (sum of the dK slots), dV = sum of the dV
// slots, in slot order, fp32 -> bf16, 4 elements per step. n4k, n4v: float4
// per dK slot and per dV slot (the dV slots follow the split dK slots).
__global__ void bwd_dkv_sum(const float* __restrict__ part, __nv_bfloat16* __restrict__ dk,
                            __nv_bfloat16* __restrict__ dv, long n4k, long n4v, int split, float scale) {
    const long stride = (long)gridDim.x * blockDim.x;
    const float4* p4 = reinterpret_cast<const float4*>(part);
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n4k + n4v; i += stride) {
        const bool is_v = i >= n4k;
        const long j = is_v ? i - n4k : i;
        const long n4 = is_v ? n4v : n4k;
        const float4* src = p4 + (is_v ? (long)split * n4k : 0) + j;
        float4 a = src[0];
        for (int sl = 1; sl < split; ++sl) {
            const float4 b = src[(long)sl * n4];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        const float mul = is_v ? 1.f : scale;
        uint2 o;
        o.x = pack_bf16x2(a.x * mul, a.y * mul);
        o.y = pack_bf16x2(a.z * mul, a.w * mul);
        reinterpret_cast<uint2*>(is_v ? dv : dk)[j] = o;
    }
}

// dQ = scale * accumulator, fp32 -> bf16, 8 elements per step.
__global__ void bwd_convert(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq, long n8, float scale) {
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
        uint4 o;
        o.x = pack_bf16x2(a.x * scale, a.y * scale);
        o.y = pack_bf16x2(a.z * scale, a.w * scale);
        o.z = pack_bf16x2(b.x * scale, b.y * scale);
        o.w = pack_bf16x2(b.z * scale, b.w * scale);
        reinterpret_cast<uint4*>(dq)[i] = o;
    }
}

// ----------------------------------------------------------------------------
// kDet: deterministic dQ accumulation (a separate instantiation keeps the
// other path's code out of each kernel); kGQA: grouped heads (bwd_tile);
// kBand: the mask is a local window other than the plain causal mask (a
// left bound, or a right bound past the diagonal) or has a block mask; the
// kernels for no mask and the causal mask keep their closed forms (a key's
// query rows run from its diagonal, or from 0, to the sequence's end).
// kSparse (with kBand only): a block mask is given, the walks skip the blocks
// it drops.
template <int HD, bool kDet, bool kGQA, bool kBand, bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
           const __grid_constant__ CUtensorMap tmDQ32, const BwdParams p, const VarlenMap* vm) {
    using Lay = BwdLayout<HD>;
    constexpr int NQS = Lay::kQStages, NDS = Lay::kDOStages;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Geometry& g = p.g;
    if (base & 1023u) {   // the swizzled operand tiles need 1024-byte alignment
        if (tid == 0) atomicCAS(p.status, kStatusOk, kStatusMisaligned);
        return;
    }
    auto bar = [&](int i) -> uint32_t { return base + Lay::kBarOff + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kMiscOff + 4);

    if (tid == 0) {
        mbar_init(bar(Lay::kKVFull), 1);
        mbar_init(bar(Lay::kKVEmpty), 1);
        for (int s = 0; s < NQS; ++s) {
            mbar_init(bar(Lay::kQFull + s), 2);   // the Q tile's bytes + the row statistics
            mbar_init(bar(Lay::kQEmpty + s), 1);
        }
        for (int s = 0; s < NDS; ++s) {
            mbar_init(bar(Lay::kDOFull + s), 1);
            mbar_init(bar(Lay::kDOEmpty + s), 1);
        }
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
        mbar_init(bar(Lay::kTDSFree), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmDO);
        tma_prefetch_desc(&tmDQ32);
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
    const int n_tiles = varlen ? vm->pre[g.B] * (kGQA ? p.split : 1) : p.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        setmaxnreg_dec<kRegsLoadMma>();
        uint32_t tile_it = 0, qc = 0;
        bool ok = true;
        float* stats = reinterpret_cast<float*>(smem + Lay::kStatOff);
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const BwdTile f = bwd_tile<kGQA, kBand, kSparse, kDet>(t, p, vmp, lane);
            if (kSparse ? f.nblk == 0 : f.m_begin >= f.m_end) continue;
            ok = warp_wait(bar(Lay::kKVEmpty), (tile_it & 1u) ^ 1u, w, lane);
            if (!ok) break;
            if (lane == 0) {
                mbar_expect_tx(bar(Lay::kKVFull), 2 * Lay::kTileBytes);
                for (int hf = 0; hf < Lay::kHalves; ++hf) {
                    tma_load_3d(base + Lay::kKOff + hf * kBox, &tmK, bar(Lay::kKVFull), hf * 64, f.h,
                                f.k_row0 + f.n * kBN);
                    tma_load_3d(base + Lay::kVOff + hf * kBox, &tmV, bar(Lay::kKVFull), hf * 64, f.h,
                                f.k_row0 + f.n * kBN);
                }
            }
            __syncwarp();
            ++tile_it;
            QWalk qw = qwalk_start<kSparse>(f, lane);
            for (int u = 0; u < f.nblk && ok; ++u, qwalk_step<kGQA, kSparse>(qw, f, lane)) {
                const int m = qw.m;
                const uint32_t st = qc % NQS;
                ok = warp_wait(bar(Lay::kQEmpty + st), ((qc / NQS) & 1u) ^ 1u, w, lane);
                if (!ok) break;
                // Q first (arrival 1 of 2 with its byte count), so the copy overlaps the
                // global loads of the row statistics below (arrival 2 of 2)
                if (lane == 0) {
                    mbar_expect_tx(bar(Lay::kQFull + st), Lay::kTileBytes);
                    for (int hf = 0; hf < Lay::kHalves; ++hf)
                        tma_load_3d(base + Lay::kQOff + st * Lay::kTileBytes + hf * kBox, &tmQ, bar(Lay::kQFull + st),
                                    hf * 64, qw.h, f.q_row0 + m * kBM);
                }
                // row statistics for this query block, negated: -lse in log2 units and -D
                float* nlse2 = stats + st * 256;
                float* ndd = nlse2 + 128;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = m * kBM + lane * 4 + e;
                    float lv = -INFINITY, dv = 0.f;   // negated; rows past the end: P = 0
                    if (r < f.lq) {
                        long si = varlen ? (long)qw.h * g.Lq + f.q_row0 + r
                                         : ((long)f.b * g.H + qw.h) * g.Lq + r;
                        lv = -p.lse[si] * kLog2e;
                        dv = -p.delta[si];
                    }
                    nlse2[lane * 4 + e] = lv;
                    ndd[lane * 4 + e] = dv;
                }
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Lay::kQFull + st));
                __syncwarp();
                const uint32_t sd = qc % NDS;
                ok = warp_wait(bar(Lay::kDOEmpty + sd), ((qc / NDS) & 1u) ^ 1u, w, lane);
                if (!ok) break;
                if (lane == 0) {
                    mbar_expect_tx(bar(Lay::kDOFull + sd), Lay::kTileBytes);
                    for (int hf = 0; hf < Lay::kHalves; ++hf)
                        tma_load_3d(base + Lay::kDOOff + sd * Lay::kTileBytes + hf * kBox, &tmDO,
                                    bar(Lay::kDOFull + sd), hf * 64, qw.h, f.q_row0 + m * kBM);
                }
                __syncwarp();
                ++qc;
            }
        }
        if (lane == 0) {
            if (tile_it) drain_wait(bar(Lay::kKVFull), (tile_it - 1) & 1u, p.wait_budget_ns);
            for (uint32_t i = 0; i < (uint32_t)NQS && i < qc; ++i) {
                const uint32_t n = qc - 1 - i;
                drain_wait(bar(Lay::kQFull + n % NQS), (n / NQS) & 1u, p.wait_budget_ns);
            }
            for (uint32_t i = 0; i < (uint32_t)NDS && i < qc; ++i) {
                const uint32_t n = qc - 1 - i;
                drain_wait(bar(Lay::kDOFull + n % NDS), (n / NDS) & 1u, p.wait_budget_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        setmaxnreg_dec<kRegsLoadMma>();
        constexpr uint32_t kIdSq = idesc_bf16_f32(kBN, kBM, false, false);    // S^T, dP^T: 128 x 128
        constexpr uint32_t kIdKV = idesc_bf16_f32(kBN, HD, false, true);      // dV, dK: 128 x d, B MN-major
        constexpr uint32_t kIdDQ = idesc_bf16_f32(kBM, HD, true, true);       // dQ: A (dS) MN-major
        // Descriptors are built once; each MMA adds a compile-time offset to the low half.
        // K-major views (d contiguous along K) and MN-major views of the same tiles.
        const SmemDesc k_km = sdesc_sw128_split(base + Lay::kKOff, 16, 1024);
        const SmemDesc v_km = sdesc_sw128_split(base + Lay::kVOff, 16, 1024);
        const SmemDesc k_mn = sdesc_sw128_split(base + Lay::kKOff, kBox, 1024);
        const SmemDesc ds_mn0 = sdesc_sw128_split(base + Lay::kDSOff, kBox, 1024);
        const SmemDesc q_km0 = sdesc_sw128_split(base + Lay::kQOff, 16, 1024);
        const SmemDesc q_mn0 = sdesc_sw128_split(base + Lay::kQOff, kBox, 1024);
        const SmemDesc do_km0 = sdesc_sw128_split(base + Lay::kDOOff, 16, 1024);
        const SmemDesc do_mn0 = sdesc_sw128_split(base + Lay::kDOOff, kBox, 1024);
        auto at_stage = [&](SmemDesc d, uint32_t stage) {   // the stage-th tile of a ring
            d.lo += stage * desc_step(Lay::kTileBytes);
            return d;
        };
        // D[128 x 128] = A[128 x d] * B[128 x d]^T, both K-major (d contiguous)
        auto mma_nt = [&](uint32_t d_tmem, SmemDesc a, SmemDesc b) {
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t off = desc_step((k >> 2) * kBox + (k & 3) * 32);
                mma_ss(d_tmem, a, off, b, off, kIdSq, k > 0);
            }
        };
        // The d = 64 order issues from the whole warp (one elected lane) in the default
        // mode (B2 H16 L8192 d64: causal 667 -> 726 TF/s, non-causal 714 -> 791) and
        // from lane 0 in the deterministic mode, where the converged issue measured
        // slower (469 -> 401). The d = 128 order issues from lane 0 (converged issue
        // measured 15-35% slower there, for reasons not found).
        auto ss = [&](uint32_t d_tmem, SmemDesc a, uint32_t a_step, SmemDesc b, uint32_t b_step, uint32_t id,
                      uint32_t acc) {
            if constexpr (kDet) {
                if (lane == 0) mma_ss(d_tmem, a, a_step, b, b_step, id, acc);
            } else {
                mma_ss_w(d_tmem, a, a_step, b, b_step, id, acc);
            }
        };
        auto ts = [&](uint32_t d_tmem, uint32_t a_tmem, SmemDesc b, uint32_t b_step, uint32_t id, uint32_t acc) {
            if constexpr (kDet) {
                if (lane == 0) mma_ts(d_tmem, a_tmem, b, b_step, id, acc);
            } else {
                mma_ts_w(d_tmem, a_tmem, b, b_step, id, acc);
            }
        };
        auto nt = [&](uint32_t d_tmem, SmemDesc a, SmemDesc b) {
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t off = desc_step((k >> 2) * kBox + (k & 3) * 32);
                ss(d_tmem, a, off, b, off, kIdSq, k > 0);
            }
        };
        uint32_t tile_it = 0, qc = 0, pc = 0, dsc = 0, dqf = 0;
        bool ok = true;
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const BwdTile f = bwd_tile<kGQA, kBand, kSparse, kDet>(t, p, vmp, lane);
            if (kSparse ? f.nblk == 0 : f.m_begin >= f.m_end) continue;
            ok = warp_wait(bar(Lay::kKVFull), tile_it & 1u, w, lane);
            if (!ok) break;
            ++tile_it;
            uint32_t st = qc % NQS;
            ok = warp_wait(bar(Lay::kQFull + st), (qc / NQS) & 1u, w, lane);
            if (!ok) break;
            tc_fence_after_sync();
            if (lane == 0) {   // S^T for the first query block
                mma_nt(tmem + Lay::kTS, k_km, at_stage(q_km0, st));
                tc_commit(bar(Lay::kSFull));
            }
            __syncwarp();
            if constexpr (Lay::kSplitDP) {
                // dP^T of the first query block right away: nothing else uses its columns
                const uint32_t sd0 = qc % NDS;
                ok = warp_wait(bar(Lay::kDOFull + sd0), (qc / NDS) & 1u, w, lane);
                if (!ok) break;
                tc_fence_after_sync();
                {
                    nt(tmem + Lay::kTDP, v_km, at_stage(do_km0, sd0));
                    if (lane == 0) tc_commit(bar(Lay::kDPFull));
                }
                __syncwarp();
                for (int u = 0; u < f.nblk; ++u) {
                    const uint32_t sd = qc % NDS, dsb = qc & 1u;   // dO stage, dS tile of this block
                    const SmemDesc q_mn = at_stage(q_mn0, st);
                    SmemDesc ds_mn = ds_mn0;
                    ds_mn.lo += dsb * desc_step(Lay::kDSBytes);
                    // dV += P^T dO (P^T from tensor memory)
                    ok = warp_wait(bar(Lay::kPFull), pc & 1u, w, lane);
                    if (!ok) break;
                    ++pc;
                    tc_fence_after_sync();
                    {
                        const SmemDesc do_mn = at_stage(do_mn0, sd);
#pragma unroll
                        for (int k = 0; k < kBM / 16; ++k)
                            ts(tmem + Lay::kTDV, tmem + Lay::kTS + packed_col(k),
                               do_mn, desc_step(k * 2048), kIdKV, (u > 0 || k > 0) ? 1u : 0u);
                        if (lane == 0) tc_commit(bar(Lay::kDOEmpty + sd));   // dO is no longer read
                    }
                    __syncwarp();
                    const bool more = u + 1 < f.nblk;
                    const uint32_t st_next = more ? (qc + 1) % NQS : st;
                    if (more) {   // S^T of the next query block over P^T (which dV has read)
                        ok = warp_wait(bar(Lay::kQFull + st_next), ((qc + 1) / NQS) & 1u, w, lane);
                        if (!ok) break;
                        tc_fence_after_sync();
                        {
                            nt(tmem + Lay::kTS, k_km, at_stage(q_km0, st_next));
                            if (lane == 0) tc_commit(bar(Lay::kSFull));
                        }
                        __syncwarp();
                    }
                    // dS^T is written and dP^T read: dP^T of the next block ahead of dK and dQ
                    ok = warp_wait(bar(Lay::kDSFull), dsc & 1u, w, lane);
                    if (!ok) break;
                    ++dsc;
                    if (more) {
                        const uint32_t sd_next = (qc + 1) % NDS;
                        ok = warp_wait(bar(Lay::kDOFull + sd_next), ((qc + 1) / NDS) & 1u, w, lane);
                        if (!ok) break;
                    }
                    tc_fence_after_sync();
                    {
                        if (more) {
                            nt(tmem + Lay::kTDP, v_km, at_stage(do_km0, (qc + 1) % NDS));
                            if (lane == 0) tc_commit(bar(Lay::kDPFull));
                        }
                        // dK += dS^T Q (dS^T from its own tensor-memory columns)
#pragma unroll
                        for (int k = 0; k < kBM / 16; ++k)
                            ts(tmem + Lay::kTDK, tmem + Lay::kTDS + packed_col_ds(k),
                               q_mn, desc_step(k * 2048), kIdKV, (u > 0 || k > 0) ? 1u : 0u);
                        if (lane == 0) tc_commit(bar(Lay::kTDSFree));
                    }
                    __syncwarp();
                    // dQ = dS K into its own columns once the previous dQ tile has left them
                    ok = warp_wait(bar(Lay::kDQFree), (dqf & 1u) ^ 1u, w, lane);
                    if (!ok) break;
                    ++dqf;
                    tc_fence_after_sync();
                    {
#pragma unroll
                        for (int k = 0; k < kBN / 16; ++k)
                            ss(tmem + Lay::kTDQ, ds_mn, desc_step(k * 2048), k_mn, desc_step(k * 2048), kIdDQ,
                               k > 0 ? 1u : 0u);
                        if (lane == 0) tc_commit(bar(Lay::kDQFull));
                        if (lane == 0) tc_commit(bar(Lay::kQEmpty + st));
                        if (!more) {
                            if (lane == 0) tc_commit(bar(Lay::kDKVFull));
                            if (lane == 0) tc_commit(bar(Lay::kKVEmpty));
                        }
                    }
                    __syncwarp();
                    ++qc;
                    st = st_next;
                }
            } else {
            for (int u = 0; u < f.nblk; ++u) {
                const uint32_t sd = qc % NDS, dsb = qc & 1u;   // dO stage, dS tile of this block
                const SmemDesc do_km = at_stage(do_km0, sd), do_mn = at_stage(do_mn0, sd);
                const SmemDesc q_mn = at_stage(q_mn0, st);
                SmemDesc ds_mn = ds_mn0;
                ds_mn.lo += dsb * desc_step(Lay::kDSBytes);
                // dP^T = V dO^T into the dP/dQ block once the previous dQ tile is read out
                ok = warp_wait(bar(Lay::kDQFree), (dqf & 1u) ^ 1u, w, lane);
                if (!ok) break;
                ++dqf;
                ok = warp_wait(bar(Lay::kDOFull + sd), (qc / NDS) & 1u, w, lane);
                if (!ok) break;
                tc_fence_after_sync();
                if (lane == 0) {
                    mma_nt(tmem + Lay::kTDP, v_km, do_km);
                    tc_commit(bar(Lay::kDPFull));
                }
                __syncwarp();
                // dV += P^T dO (P^T from tensor memory)
                ok = warp_wait(bar(Lay::kPFull), pc & 1u, w, lane);
                if (!ok) break;
                ++pc;
                tc_fence_after_sync();
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < kBM / 16; ++k)
                        mma_ts(tmem + Lay::kTDV, tmem + Lay::kTS + packed_col(k),
                               do_mn, desc_step(k * 2048), kIdKV, (u > 0 || k > 0) ? 1u : 0u);
                    tc_commit(bar(Lay::kDOEmpty + sd));   // dO is no longer read
                }
                __syncwarp();
                const bool more = u + 1 < f.nblk;
                const uint32_t st_next = more ? (qc + 1) % NQS : st;
                // S^T of the next query block right after dV, ahead of dK/dQ: it overwrites
                // P^T, which dV (issued before it) has consumed, and the compute warps
                // find it ready when they finish this block's dS^T. (Issued after dK/dQ
                // it made them wait for three products: d = 128 backward 772 -> 800 TF/s
                // non-causal, d = 64 462 -> 539 causal.)
                if (more) {
                    ok = warp_wait(bar(Lay::kQFull + st_next), ((qc + 1) / NQS) & 1u, w, lane);
                    if (!ok) break;
                    tc_fence_after_sync();
                    if (lane == 0) {
                        mma_nt(tmem + Lay::kTS, k_km, at_stage(q_km0, st_next));
                        tc_commit(bar(Lay::kSFull));
                    }
                    __syncwarp();
                }
                // dK += dS^T Q (dS^T from tensor memory) and dQ = dS K (dS from shared memory)
                ok = warp_wait(bar(Lay::kDSFull), dsc & 1u, w, lane);
                if (!ok) break;
                ++dsc;
                tc_fence_after_sync();
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < kBM / 16; ++k)
                        mma_ts(tmem + Lay::kTDK, tmem + Lay::kTDS + packed_col(k),
                               q_mn, desc_step(k * 2048), kIdKV, (u > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                    for (int k = 0; k < kBN / 16; ++k)
                        mma_ss(tmem + Lay::kTDQ, ds_mn, desc_step(k * 2048), k_mn, desc_step(k * 2048), kIdDQ,
                               k > 0 ? 1u : 0u);
                    tc_commit(bar(Lay::kDQFull));
                    tc_commit(bar(Lay::kQEmpty + st));
                    if (!more) {
                        tc_commit(bar(Lay::kDKVFull));
                        tc_commit(bar(Lay::kKVEmpty));
                    }
                }
                __syncwarp();
                ++qc;
                st = st_next;
            }
            }
        }
        if (lane == 0) {
            tc_commit(bar(Lay::kDrain));
            drain_wait(bar(Lay::kDrain), 0, p.wait_budget_ns);
        }
        __syncwarp();
    } else if (warp < 4) {
        setmaxnreg_dec<kRegsLoadMma>();   // idle warps of the load/MMA warpgroup
    } else if (warp < 12) {
        // ------------------------------------------------------------ compute warpgroups
        const int wg = (warp - 4) >> 2;            // query columns [64*wg, 64*wg + 64)
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;         // key row inside the block
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = g.scale_log2;
        uint8_t* const ds_tiles = smem + Lay::kDSOff + wg * kBox;   // this warpgroup's 64 query columns
        const float* stats = reinterpret_cast<const float*>(smem + Lay::kStatOff);
        uint32_t sc = 0, qc = 0, dpc = 0, dsw = 0, tile_it = 0, tds = 0;
        bool ok = true;
        uint32_t rr[32];
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const BwdTile f = bwd_tile<kGQA, kBand, kSparse, kDet>(t, p, vmp, lane);
            const int key = f.n * kBN + r;
            const bool key_ok = key < f.lk;
            const long krow = (long)f.k_row0 + key;
            // this thread's dK/dV row: bf16 outputs, or (split tiles) fp32 partial
            // slots, dK slot f.s and dV slot split + f.s; computed where used, so
            // that no pointer stays live through the query-block loop
            const bool partial = kGQA && p.split > 1;
            auto kv_off = [&]() { return (krow * g.Hkv + f.h) * HD + wg * (HD / 2); };
            auto part_slot = [&](int which) {   // 0: dV, 1: dK
                const long slot = (varlen ? (long)g.Lk : (long)g.B * g.Lk) * g.Hkv * HD;
                return p.dkv_part + (which ? f.s : p.split + f.s) * slot + kv_off();
            };
            if (kSparse ? f.nblk == 0 : f.m_begin >= f.m_end) {   // no query sees this key block
                __nv_bfloat16* dv_ptr = p.dv + kv_off();
                __nv_bfloat16* dk_ptr = p.dk + kv_off();
                float* pk_ptr = partial ? part_slot(1) : nullptr;
                float* pv_ptr = partial ? part_slot(0) : nullptr;
                if (key_ok) {
                    if (partial) {
                        for (int c = 0; c < HD / 8; ++c) {
                            reinterpret_cast<float4*>(pv_ptr)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                            reinterpret_cast<float4*>(pk_ptr)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < HD / 16; ++c) {
                            reinterpret_cast<uint4*>(dv_ptr)[c] = make_uint4(0, 0, 0, 0);
                            reinterpret_cast<uint4*>(dk_ptr)[c] = make_uint4(0, 0, 0, 0);
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
            QWalk qw = qwalk_start<kSparse>(f, lane);
            for (int u = 0; u < f.nblk; ++u, qwalk_step<kGQA, kSparse>(qw, f, lane)) {
                const int m = qw.m;
                const uint32_t st = qc % NQS;
                uint8_t* ds_tile = ds_tiles + (qc & 1u) * Lay::kDSBytes;   // alternate dS tiles per block
                ok = warp_wait(bar(Lay::kSFull), sc & 1u, w, lane);
                if (!ok) break;
                ++sc;
                ok = warp_wait(bar(Lay::kQFull + st), (qc / NQS) & 1u, w, lane);   // stats visibility
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
                // the producer stages -lse (log2 units) and -D, so both steps are packed fp32 pairs
                const float* nlse2 = stats + st * 256 + wg * 64;
                const float* ndd = stats + st * 256 + 128 + wg * 64;
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
                ok = warp_wait(bar(Lay::kDSEmpty + (dsw & 1u)), ((dsw >> 1) & 1u) ^ 1u, w, lane);
                if (!ok) break;
                ++dsw;
                uint32_t ds2[32];   // dS^T, two bf16 per word
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
                if constexpr (Lay::kSplitDP) {
                    // dS^T into its own columns once dK has read the previous one
                    if (tds > 0) {
                        ok = warp_wait(bar(Lay::kTDSFree), (tds - 1) & 1u, w, lane);
                        if (!ok) break;
                        tc_fence_after_sync();
                    }
                    ++tds;
                    tmem_st32(tmem + lane_off + Lay::kTDS + wg * 32, ds2);
                } else {
                    // dS^T also into tensor memory (over this warpgroup's dP^T columns, already read) for dK
                    tmem_st32(tmem + lane_off + Lay::kTDS + wg * 64, ds2);
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(bar(Lay::kDSFull));
            }
            if (!ok) break;
            // epilogue: this warpgroup writes d/2 columns of dV and of dK for its key row
            ok = warp_wait(bar(Lay::kDKVFull), tile_it & 1u, w, lane);
            if (!ok) break;
            ++tile_it;
            tc_fence_after_sync();
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t col0 = (which ? Lay::kTDK : Lay::kTDV) + wg * (HD / 2);
                const float mul = which ? g.scale : 1.f;
                __nv_bfloat16* dst = (which ? p.dk : p.dv) + kv_off();
                float* pdst = partial ? part_slot(which) : nullptr;
#pragma unroll
                for (int c = 0; c < HD / 64; ++c) {
                    tmem_ld32(tmem + lane_off + col0 + c * 32, rr);
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
        // Each dQ tile (128 query rows x d, fp32) goes from tensor memory to the
        // global accumulator: staged through shared memory (the dS^T tile this
        // block's dQ MMA has read) and added by TMA reduce-adds, each warp its own
        // 32 rows (dq_reduce.cuh). Deterministic mode: the same reduce-adds under
        // the tile's semaphore, in key-block order, every warp's completing before
        // the next block's start.
        const int quarter = warp & 3;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        setmaxnreg_inc<kRegsDq>();
        const bool leader = warp == 12 && lane == 0;
        uint32_t dqc = 0, sgo = 0, rdc = 0;
        bool ok = true;
        uint32_t rr[32];
        // Deterministic mode: the turn of the block's dQ tile. The leader waits for it and
        // tells the warpgroup, whose lanes all wait on that barrier. At d = 128 the turn is
        // taken before the dQ tile is ready, so the wait overlaps the dQ product instead of
        // following it (B1 H32 L32768 causal 641 -> 731 TF/s, B4 H16 L4096 non-causal 517 ->
        // 593); the d = 64 order keeps it after (463 -> 443 taken before).
        constexpr bool kEarlyTurn = !Lay::kSplitDP;
        int* sem = nullptr;
        auto take_turn = [&](const BwdTile& ft, int h, int m) -> bool {
            sem = p.semaphores + dq_semaphore(p, ft, h, m, varlen);
            if (leader) {
                if (sem_wait(sem, dq_turn<kBand, kSparse>(p, ft, h, m), w)) fence_proxy_async_global();
                mbar_arrive(bar(Lay::kSemGo));   // arrive even after a failure; abort_flag tells
            }
            const bool go = warp_wait(bar(Lay::kSemGo), sgo & 1u, w, lane);
            ++sgo;
            return go && !*abort_flag;
        };
        for (int k = 0, t = blockIdx.x; t < n_tiles && ok; t = snake_tile(blockIdx.x, ++k, gridDim.x)) {
            const BwdTile f = bwd_tile<kGQA, kBand, kSparse, kDet>(t, p, vmp, lane);
            QWalk qw = qwalk_start<kSparse>(f, lane);
            for (int u = 0; u < f.nblk; ++u, qwalk_step<kGQA, kSparse>(qw, f, lane)) {
                const int m = qw.m;
                if constexpr (kDet && kEarlyTurn) {
                    ok = take_turn(f, qw.h, m);
                    if (!ok) break;
                }
                ok = warp_wait(bar(Lay::kDQFull), dqc & 1u, w, lane);
                if (!ok) break;
                // the dS tile this block's dQ MMA read is free now: stage dQ through it
                const uint32_t dsb = dqc & 1u;
                uint8_t* stage = smem + Lay::kDSOff + dsb * Lay::kDSBytes;
                const uint32_t stage_s = base + Lay::kDSOff + dsb * Lay::kDSBytes;
                ++dqc;
                tc_fence_after_sync();
                if constexpr (kDet && !kEarlyTurn) {
                    ok = take_turn(f, qw.h, m);
                    if (!ok) break;
                }
                // the whole dQ row leaves tensor memory at once, so the next dP^T can start
                // (deterministic mode: once the semaphore has let this block in)
                uint32_t row[HD];
                if constexpr (HD == 128) {
                    tmem_ld128(tmem + lane_off + Lay::kTDQ, row);
                } else {
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) {
                        tmem_ld32(tmem + lane_off + Lay::kTDQ + c * 32, rr);
#pragma unroll
                        for (int i = 0; i < 32; ++i) row[c * 32 + i] = rr[i];
                    }
                }
                tc_fence_before_sync();
                mbar_arrive(bar(Lay::kDQFree));
                dq_warp_reduce(&tmDQ32, stage, stage_s, row, HD / 64, 0, qw.h, f.q_row0 + m * kBM, quarter, lane);
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
                    // every warp's adds of this block are complete: the next block's turn
                    if (leader && mbar_wait(bar(Lay::kRedDone), rdc & 1u, w))
                        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sem) : "memory");
                    ++rdc;
                }
                __syncwarp();
            }
        }
        if (lane == 0) bulk_wait_group0();   // the last reduce-adds complete before the CTA exits
    }
    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// The instantiation for a mask: none or causal; a general band; a band with a block mask.
template <int HD, bool kDet, bool kGQA>
auto bwd_kernel_for(bool band, bool sparse) {
    return sparse ? bwd_kernel<HD, kDet, kGQA, true, true>
                  : (band ? bwd_kernel<HD, kDet, kGQA, true, false> : bwd_kernel<HD, kDet, kGQA, false, false>);
}

template <int HD>
cudaError_t launch_bwd_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const PairMaps& pm, bool pair,
                          const BwdParams& p, int num_sms, cudaStream_t stream) {
    const Geometry& g = p.g;
    const bool varlen = g.cu_seqlens != nullptr;
    const long rows_q = varlen ? (long)g.Lq : (long)g.B * g.Lq;
    const long n_acc4 = rows_q * g.H * HD / 4;
    const int n_sem = (int)bwd_semaphore_count(g.B, g.H, g.Lq, varlen);
    // the varlen map lives right after the semaphores
    VarlenMap* vm = reinterpret_cast<VarlenMap*>(
        reinterpret_cast<char*>(p.semaphores) + (((size_t)n_sem * sizeof(int) + 255) & ~(size_t)255));
    {
        const long work = rows_q * g.H * 8;   // eight lanes per (row, head)
        int blocks = (int)((work + 255) / 256);
        if (blocks > 8 * num_sms) blocks = 8 * num_sms;
        if (blocks < 1) blocks = 1;
        bwd_prep<<<blocks, 256, 0, stream>>>(p, vm, rows_q, n_acc4, n_sem, pair ? 2 * kBN : kBN);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaSuccess;
    // Q and dO bytes of every query head: the working set of a global walk
    const double ws_bytes = 2.0 * 2.0 * (double)rows_q * g.H * HD;
    if (pair) {
        BwdParams pp = p;   // work tiles are key-block pairs
        pp.nm = bwd_pair_tiles_per_head(g.Lk);
        pp.n_tiles = varlen ? 0 : g.B * g.Hkv * pp.nm;   // a tile walks every query head of its group
        pp.sections = sched_sections_pay(g.B, g.Hkv, pp.nm, p.head_section, 1, num_sms / 2, ws_bytes) ? 1 : 0;
        e = launch_bwd_pair(pm, tk, tv, pp, vm, num_sms, stream);
        if (e != cudaSuccess) return e;
    } else if constexpr (HD > 128) {
        e = launch_bwd_wide(tq, tk, tv, tdo, pm.dq32, p, vm, num_sms, stream);
        if (e != cudaSuccess) return e;
    } else {
        using Lay = BwdLayout<HD>;
        const bool gqa = g.group > 1, sparse = p.mask.ptr != nullptr;
        const bool band = sparse || g.win_left >= 0 || g.win_right > 0;
        auto kern = p.deterministic ? (gqa ? bwd_kernel_for<HD, true, true>(band, sparse)
                                           : bwd_kernel_for<HD, true, false>(band, sparse))
                                    : (gqa ? bwd_kernel_for<HD, false, true>(band, sparse)
                                           : bwd_kernel_for<HD, false, false>(band, sparse));
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        // the register split re-distributes exactly the registers the CTA launches with
        if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
        const int grid = varlen ? num_sms : min(p.n_tiles, num_sms);
        BwdParams pk = p;
        pk.sections = sched_sections_pay(g.B, g.Hkv, p.nm, p.head_section, gqa ? p.split : 1, grid, ws_bytes) ? 1 : 0;
        if (grid > 0) {
            kern<<<grid, kThreads, Lay::kSmemBytes, stream>>>(tq, tk, tv, tdo, pm.dq32, pk, vm);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
    }
    if (p.split > 1 && !pair) {   // (the pair kernel writes dK and dV of the whole group itself)
        const long rows_k = varlen ? (long)g.Lk : (long)g.B * g.Lk;
        const long n4k = rows_k * g.Hkv * HD / 4, n4v = rows_k * g.Hkv * p.d_v / 4;
        int blocks = (int)((n4k + n4v + 255) / 256);
        if (blocks > 8 * num_sms) blocks = 8 * num_sms;
        if (blocks < 1) blocks = 1;
        bwd_dkv_sum<<<blocks, 256, 0, stream>>>(p.dkv_part, p.dk, p.dv, n4k, n4v, p.split, g.scale);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const long n8 = rows_q * g.H * HD / 8;
        int blocks = (int)((n8 + 255) / 256);
        if (blocks > 8 * num_sms) blocks = 8 * num_sms;
        if (blocks < 1) blocks = 1;
        bwd_convert<<<blocks, 256, 0, stream>>>(p.dq_acc, p.dq, n8, g.scale);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

size_t bwd_varlen_map_bytes() { return sizeof(VarlenMap); }

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const PairMaps& pm, bool pair,
                       const BwdParams& p, int num_sms, cudaStream_t stream) {
    pair = pair && bwd_pair_supported(p);
    switch (p.g.d) {
        case 64: return launch_bwd_hd<64>(tq, tk, tv, tdo, tdq, pm, pair, p, num_sms, stream);
        case 128: return launch_bwd_hd<128>(tq, tk, tv, tdo, tdq, pm, pair, p, num_sms, stream);
        case 192: return launch_bwd_hd<192>(tq, tk, tv, tdo, tdq, pm, false, p, num_sms, stream);
        case 256: return launch_bwd_hd<256>(tq, tk, tv, tdo, tdq, pm, false, p, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
