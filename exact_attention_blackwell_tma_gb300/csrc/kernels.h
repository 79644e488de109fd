// Internal interface between the C-ABI host layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Problem geometry as the kernels see it. Rows are "packed": a dense tensor
// [B, L, H, d] is viewed as [B*L, H, d], batch b starting at packed row b*L;
// a varlen tensor [T, H, d] has sequence b starting at cu_seqlens[b].
// Grouped heads: q, o, dO, dq have H heads, k, v, dk, dv have Hkv; query head
// h reads key/value head h / group (group = H / Hkv; 1 for multi-head).
struct Geometry {
    int B, H, Lq, Lk, d;      // dense: sizes; varlen: Lq, Lk = packed query and key rows
    int Hkv, group;           // key/value heads, query heads per key/value head
    int causal;               // the mask has a right bound (win_right >= 0): longest-first walks
    int win_left, win_right;  // mask band (mask.cuh): keys i + delta - win_left .. i + delta + win_right
                              // of query i, -1: no bound on that side; causal is win_right = 0
    float scale;              // softmax scale (> 0)
    float scale_log2;         // scale * log2(e)
    const int* cu_seqlens;    // device, B+1 query offsets, or null (dense)
    const int* cu_seqlens_k;  // device, B+1 key offsets (varlen; cu_seqlens when they are shared)
};

// A block mask (dense problems): bytes [heads][ceil(Lq/128)][ceil(Lk/128)],
// heads 1 (shared) or H; a zero byte drops that 128 x 128 block (mask.cuh).
// ptr null: none.
struct BlockMask {
    const unsigned char* ptr;
    int heads;
};
__host__ __device__ inline int mask_rows(const Geometry& g) { return (g.Lq + 127) / 128; }
__host__ __device__ inline int mask_cols(const Geometry& g) { return (g.Lk + 127) / 128; }

// The fields are ordered to leave no padding: with more than 128 bytes of
// parameters the forward kernel's register allocation spilled more.
struct FwdParams {
    Geometry g;
    __nv_bfloat16* o;         // rows and heads of q, head dim dv
    float* lse;               // dense [B, H, Lq]; varlen [H, T]
    int* status;
    uint64_t wait_budget_ns;
    int dv;                   // head dim of v and o (g.d for q and k)
    int n_tiles;              // dense: exact count; varlen: computed on device
    int nm;                   // dense: query blocks per (b, h): 256 rows (d <= 128) or 128 rows
    int head_section;         // heads per L2 section (LPT walk)
    BlockMask mask;
};
static_assert(sizeof(FwdParams) <= 128, "forward parameters");

struct BwdParams {
    Geometry g;
    const __nv_bfloat16* o;
    const __nv_bfloat16* dout;
    const float* lse;         // natural-log LSE from the forward, layout as FwdParams::lse
    float* dq_acc;            // fp32 accumulator, layout of q
    float* delta;             // D_i = rowsum(dO * O), layout of lse
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int* semaphores;          // deterministic mode: two counters per dQ tile (one per column chunk)
    float* dkv_part;          // split > 1: fp32 partial dK (slots 0..split-1, each laid out like k),
                              // then partial dV (slots laid out like v); null otherwise
    int split;                // tiles per key block of a key/value head (divides g.group)
    int d_v;                  // head dim of v, o, dO, dv (g.d, or 128 with g.d = 192)
    int deterministic;
    int n_tiles;              // dense: exact count, split included
    int nm;                   // dense: 128-row K/V blocks per (b, h)
    int nq;                   // dense: 128-row Q blocks per (b, h)
    int head_section;
    int sections;             // causal dense, default mode: walk heads in sections (sched_sections_pay)
    int* status;
    uint64_t wait_budget_ns;
    BlockMask mask;
};

// Semaphores of the deterministic backward: two per dQ tile (one per dQ column
// chunk of the wide kernel). A varlen sequence b starting at packed row s has
// its query block m at index s/128 + b + m < T/128 + B + 1 within a head.
// The host layer sizes the workspace and the launcher places the varlen map
// after the semaphores with this one count.
inline long bwd_semaphore_count(int B, int H, int Lq, bool varlen) {
    return 2L * (varlen ? (long)H * (Lq / 128 + B + 1) : (long)B * H * ((Lq + 127) / 128));
}

// Grouped heads in the backward: a work tile is one 128-key block of one
// key/value head and the query heads of its group that it visits. With one
// tile per key block a problem with few key/value heads has too few tiles to
// balance the SMs (the longest tile carries the whole group's longest rows),
// so the group's query heads are split over `split` tiles, split the smallest
// divisor of the group that gives at least kSplitTargetTiles tiles (a fixed
// target, about four per SM, so the workspace depends on the sizes alone).
// Split tiles write fp32 partial dK and dV to slots of their own, which a last
// kernel sums in slot order: the result is the same on every run.
constexpr long kSplitTargetTiles = 640;
inline int bwd_head_split(int B, int Hkv, int group, int Lk, bool varlen) {
    const long kblocks = varlen ? (Lk + 127) / 128 : (long)B * ((Lk + 127) / 128);
    const long tiles = kblocks * Hkv;
    for (int s = 1; s < group; ++s)
        if (group % s == 0 && tiles * s >= kSplitTargetTiles) return s;
    return group > 0 ? group : 1;
}
// Bytes of the partial dK/dV slots for a split (0 when split == 1); dv: head dim of v.
inline size_t bwd_partial_bytes(int split, long rows_k, int Hkv, int d, int dv) {
    return split > 1 ? (size_t)split * rows_k * Hkv * (d + dv) * sizeof(float) : 0;
}

// Launchers (return cudaSuccess or the launch error).
// poly_every: exp2 emulation of the plain kernel (no left window bound, no
// block mask): 0 (MUFU only), 8 or 4 (one column pair in every 8 or 4 by the
// FMA polynomial).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int poly_every, int num_sms, cudaStream_t stream);
// Head dims 192 and 256 (and d_qk = 192 with d_v = 128): one 128-row Q tile per
// work tile (nm counts 128-row blocks).
cudaError_t launch_fwd_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, int num_sms, cudaStream_t stream);
// Tensor maps with boxes of fewer rows or columns: q and dO in 64-row x
// 64-column bf16 boxes (the CTA-pair backward), and the dQ accumulator in 32-row
// x 32-column fp32 boxes (each dQ warp adds its own 32 rows, dq_reduce.cuh).
// q32, do32, k32: 128-row x 32-column bf16 boxes with the 64-byte swizzle, the
// pair backward's column halves at head dim 64 (encoded for that case only).
struct PairMaps {
    CUtensorMap q64, do64, dq32;
    CUtensorMap q32, do32, k32;
};
// pair: run the main kernel on CTA pairs when bwd_pair_supported(p) holds.
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq_acc, const PairMaps& pm, bool pair,
                       const BwdParams& p, int num_sms, cudaStream_t stream);

// The backward's main kernel on CTA pairs (2-CTA tensor cores, bwd_pair.cu):
// head dim 64 or 128 (q, k, v alike), grouped heads (a tile walks the query
// heads of its key/value head's group), no window beyond the causal mask, no
// block mask; dense or packed, deterministic or not.
bool bwd_pair_supported(const BwdParams& p);
// key-block pairs per (batch, head) of Lk keys
int bwd_pair_tiles_per_head(int Lk);
cudaError_t launch_bwd_pair(const PairMaps& pm, const CUtensorMap& tk, const CUtensorMap& tv, const BwdParams& p,
                            const void* varlen_map, int num_sms, cudaStream_t stream);

// Main kernel of the backward for head dims 192 and 256 (preprocess and dQ
// conversion are shared with the d <= 128 path). tdq_acc: the dQ accumulator in
// 32-row x 32-column boxes. varlen_map: the VarlenMap the preprocess kernel
// builds in the workspace (read only for varlen problems).
cudaError_t launch_bwd_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq_acc, const BwdParams& p,
                            const void* varlen_map, int num_sms, cudaStream_t stream);

int* device_status_word();   // address of the module's device status word

}  // namespace attn
