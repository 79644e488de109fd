// C-ABI host layer of libattn.so: argument checks, TMA descriptors, launches.
// The operation and the layouts are specified in include/attn.h.
#include <attn.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "kernels.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace attn {

// Device status word: kernels set it (atomically) when a bounded wait runs
// out; attn_check_status reads and clears it.
__device__ int g_attn_status;

namespace {

thread_local char g_err[512];

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = '\0';
    return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [rows, H, d] bf16 viewed as 3-D (d innermost); boxes of box_rows rows x 1
// head x 64 columns (128 bytes) with the 128-byte swizzle the MMA descriptors
// expect, or (narrow) 32 columns (64 bytes) with the 64-byte swizzle. Rows past
// `rows` read as zero.
bool make_map(CUtensorMap* m, const void* ptr, long rows, int H, int d, int box_rows = 128, bool narrow = false) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {narrow ? 32u : 64u, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The fp32 dQ accumulator [rows, H, d] for TMA reduce-adds: boxes of box_rows
// rows x 32 columns (128 bytes) with the 128-byte swizzle. Rows past `rows` are
// skipped.
bool make_map_f32(CUtensorMap* m, void* ptr, long rows, int H, int d, int box_rows = 128) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4};
    cuuint32_t box[3] = {32, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct DevInfo {
    int sms = 0;
    int* status = nullptr;
};

bool device_info(DevInfo* out) {
    static std::mutex mu;
    static DevInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    DevInfo& di = cache[dev];
    if (di.sms == 0) {
        int sms = 0;
        void* st = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        if (cudaGetSymbolAddress(&st, g_attn_status) != cudaSuccess) return false;
        di.status = static_cast<int*>(st);
        di.sms = sms;
    }
    *out = di;
    return true;
}

uint64_t wait_budget_ns() {
    static uint64_t ns = [] {
        const char* e = getenv("ATTN_WAIT_BUDGET_MS");
        double ms = e ? atof(e) : 2000.0;
        if (!(ms > 0)) ms = 2000.0;
        return (uint64_t)(ms * 1e6);
    }();
    return ns;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// exp2 emulation of the forward kernel per head dim (index 0: d = 64, 1: d =
// 128): 0 = MUFU only, 8 or 4 = one score-column pair in every 8 or 4 by the
// FMA polynomial. Set by attn_set_exp2_emulation; the defaults are the faster
// setting measured on GB300 for each head dim.
std::atomic<int> g_poly_every[2] = {{0}, {0}};

// Backward main kernel on CTA pairs (2-CTA tensor cores) where it applies; set
// by attn_set_backward_cta_pairs; the default is the faster one measured on GB300.
std::atomic<int> g_bwd_pairs{0};

// Heads per L2 section for the LPT walk: the two bf16 tensors every tile of a
// head streams (K and V in the forward, Q and dO in the backward) should fit
// in about half of the 129 MB L2 (FlashAttention-4 paper, Section 3.3).
// `rows` is the rows of those tensors per walked head.
int head_section(int H, long rows, int d) {
    const double budget = 64.0 * 1024 * 1024;
    double per_head = 2.0 * 2.0 * (double)rows * d;   // two tensors, bf16
    int hs = per_head > 0 ? (int)(budget / per_head) : H;
    if (hs < 1) hs = 1;
    if (hs > H) hs = H;
    return hs;
}

// cu_k: the key offsets of a varlen problem (== cu when one array serves both,
// which needs Lq == Lk == T).
int check_common(int B, int H, int Lq, int Lk, int d, float scale, const int* cu, const int* cu_k) {
    if (B < 0 || H <= 0 || Lq < 0 || Lk < 0) return fail(ATTN_ERR_ARG, "bad sizes B=%d H=%d Lq=%d Lk=%d", B, H, Lq, Lk);
    if (d != 64 && d != 128 && d != 192 && d != 256)
        return fail(ATTN_ERR_ARG, "head dim %d not supported (64, 128, 192, 256)", d);
    if (!std::isfinite(scale) || !(scale > 0.f)) return fail(ATTN_ERR_ARG, "scale must be finite and > 0");
    if (cu) {
        if (!cu_k) return fail(ATTN_ERR_ARG, "varlen: null key offsets");
        if (cu_k == cu && Lq != Lk)
            return fail(ATTN_ERR_ARG, "varlen: Lq and Lk must both be the packed row count T");
        if (B < 1 || B > kMaxVarlenBatch) return fail(ATTN_ERR_ARG, "varlen: B must be in [1, %d]", kMaxVarlenBatch);
    }
    long rows_q = cu ? (long)Lq : (long)B * Lq, rows_k = cu ? (long)Lk : (long)B * Lk;
    if (rows_q >= (1L << 31) || rows_k >= (1L << 31)) return fail(ATTN_ERR_ARG, "too many rows");
    return ATTN_OK;
}

int check_block_mask(const unsigned char* mask, int heads, int H, const int* cu) {
    if (!mask) return ATTN_OK;
    if (cu) return fail(ATTN_ERR_ARG, "block masks are for dense problems (cu_seqlens must be null)");
    if (heads != 1 && heads != H) return fail(ATTN_ERR_ARG, "block mask heads %d must be 1 or H = %d", heads, H);
    return ATTN_OK;
}

int check_window(int wl, int wr) {
    if (wl < -1 || wr < -1) return fail(ATTN_ERR_ARG, "window bounds must be >= 0, or -1 for none (%d, %d)", wl, wr);
    return ATTN_OK;
}

// causal != 0 sets the right bound to 0 (whatever window_right says)
void set_mask(Geometry* g, int causal, int wl, int wr) {
    g->win_left = wl;
    g->win_right = causal ? 0 : wr;
    g->causal = g->win_right >= 0 ? 1 : 0;
}

int check_heads(int H, int Hkv) {
    if (Hkv < 1 || Hkv > H || H % Hkv != 0)
        return fail(ATTN_ERR_ARG, "key/value heads %d must divide the query heads %d", Hkv, H);
    return ATTN_OK;
}

}  // namespace

int* device_status_word() {
    DevInfo di;
    return device_info(&di) ? di.status : nullptr;
}

}  // namespace attn

using namespace attn;

namespace {

// The forward behind every entry point: dense (cu_seqlens null), varlen with
// one offset array (cu_seqlens_k == cu_seqlens) or with key offsets of their own.
int fwd_entry(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int Lq,
              int Lk, int d, int dv, float scale, int causal, int window_left, int window_right,
              const unsigned char* block_mask, int mask_heads, const int* cu_seqlens, const int* cu_seqlens_k,
              cudaStream_t stream) {
    int rc = check_common(B, H, Lq, Lk, d, scale, cu_seqlens, cu_seqlens_k);
    if (rc) return rc;
    rc = check_block_mask(block_mask, mask_heads, H, cu_seqlens);
    if (rc) return rc;
    rc = check_window(window_left, window_right);
    if (rc) return rc;
    rc = check_heads(H, Hkv);
    if (rc) return rc;
    if (dv != d && !(d == 192 && dv == 128))
        return fail(ATTN_ERR_ARG, "head dims d=%d, dv=%d not supported (dv = d, or d = 192 with dv = 128)", d, dv);
    const long rows_q = cu_seqlens ? (long)Lq : (long)B * Lq;
    const long rows_k = cu_seqlens ? (long)Lk : (long)B * Lk;
    if (rows_q == 0) return ok();   // nothing to compute; pointers may be null
    if (!q || !o || !lse || (rows_k > 0 && (!k || !v))) return fail(ATTN_ERR_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return fail(ATTN_ERR_ALIGN, "tensor pointers must be 16-byte aligned");
    DevInfo di;
    if (!device_info(&di)) return fail(ATTN_ERR_LAUNCH, "cannot query the current device");
    FwdParams p{};
    p.g.B = B;
    p.g.H = H;
    p.g.Lq = Lq;
    p.g.Lk = Lk;
    p.g.d = d;
    p.g.Hkv = Hkv;
    p.g.group = H / Hkv;
    p.g.cu_seqlens = cu_seqlens;
    p.g.cu_seqlens_k = cu_seqlens ? cu_seqlens_k : nullptr;
    set_mask(&p.g, causal, window_left, window_right);
    p.g.scale = scale;
    p.g.scale_log2 = scale * kLog2e;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.dv = dv;
    p.mask.ptr = block_mask;
    p.mask.heads = mask_heads;
    p.lse = lse;
    // d <= 128: a work tile is two 128-row Q tiles; wider heads: one
    const bool wide = d > 128;
    const int rows_per_tile = wide ? 128 : 256;
    p.nm = (Lq + rows_per_tile - 1) / rows_per_tile;
    p.n_tiles = cu_seqlens ? 0 : B * H * p.nm;
    // the query heads of a group share their K and V in L2
    p.head_section = head_section(H, (cu_seqlens ? (rows_k / B) : Lk) / p.g.group, d);
    p.status = di.status;
    p.wait_budget_ns = wait_budget_ns();
    CUtensorMap tq, tk, tv;
    // a problem with no keys still needs valid descriptors: point them at q
    const long krows = rows_k > 0 ? rows_k : rows_q;
    const void* kp = rows_k > 0 ? k : q;
    const void* vp = rows_k > 0 ? v : q;
    // (a problem with no keys maps v like q, so its width must be d there)
    // (q has at least as many heads as k and v, so a view of it with Hkv heads is in bounds)
    if (!make_map(&tq, q, rows_q, H, d) || !make_map(&tk, kp, krows, Hkv, d) ||
        !make_map(&tv, vp, krows, Hkv, rows_k > 0 ? dv : d))
        return fail(ATTN_ERR_LAUNCH, "cuTensorMapEncodeTiled failed");
    const int poly = d == 64 ? g_poly_every[0].load() : (d == 128 ? g_poly_every[1].load() : 0);
    cudaError_t e = wide ? launch_fwd_wide(tq, tk, tv, p, di.sms, stream)
                         : launch_fwd(tq, tk, tv, p, poly, di.sms, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "forward launch failed: %s", cudaGetErrorString(e));
    return ok();
}

}  // namespace

extern "C" int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                            int Hkv, int Lq, int Lk, int d, int dv, float scale, int causal,
                            const int* cu_seqlens, cudaStream_t stream) {
    return fwd_entry(q, k, v, o, lse, B, H, Hkv, Lq, Lk, d, dv, scale, causal, -1, -1, nullptr, 1, cu_seqlens,
                     cu_seqlens, stream);
}

extern "C" int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                           int Lq, int Lk, int d, int d_v, float scale, int causal, int window_left,
                           int window_right, const unsigned char* block_mask, int mask_heads,
                           const int* cu_seqlens_q, const int* cu_seqlens_k, cudaStream_t stream) {
    if (cu_seqlens_k && !cu_seqlens_q) return fail(ATTN_ERR_ARG, "attn_fwd_ex: key offsets without query offsets");
    return fwd_entry(q, k, v, o, lse, B, H, Hkv, Lq, Lk, d, d_v, scale, causal, window_left, window_right,
                     block_mask, mask_heads, cu_seqlens_q, cu_seqlens_k ? cu_seqlens_k : cu_seqlens_q, stream);
}

extern "C" int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                               int Hkv, int Tq, int Tk, int d, int dv, float scale, int causal,
                               const int* cu_seqlens_q, const int* cu_seqlens_k, cudaStream_t stream) {
    if (!cu_seqlens_q || !cu_seqlens_k) return fail(ATTN_ERR_ARG, "attn_fwd_varlen: null offsets");
    return fwd_entry(q, k, v, o, lse, B, H, Hkv, Tq, Tk, d, dv, scale, causal, -1, -1, nullptr, 1, cu_seqlens_q,
                     cu_seqlens_k, stream);
}

extern "C" int attn_fwd_hdim(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                             int Lq, int Lk, int d, int dv, float scale, int causal, const int* cu_seqlens,
                             cudaStream_t stream) {
    return attn_fwd_gqa(q, k, v, o, lse, B, H, H, Lq, Lk, d, dv, scale, causal, cu_seqlens, stream);
}

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Lq,
                        int Lk, int d, float scale, int causal, const int* cu_seqlens, cudaStream_t stream) {
    return attn_fwd_gqa(q, k, v, o, lse, B, H, H, Lq, Lk, d, d, scale, causal, cu_seqlens, stream);
}

namespace {

struct BwdWorkspace {
    size_t dq_off, delta_off, part_off, sem_off, total;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// dQ accumulator | D terms | partial dK/dV slots (split grouped heads) |
// semaphores | varlen map (placed by the launcher right after the semaphores)
BwdWorkspace bwd_layout(int B, int H, int Hkv, int Lq, int Lk, int d, int dv, bool varlen) {
    BwdWorkspace w{};
    const size_t rows_q = varlen ? (size_t)Lq : (size_t)B * Lq;
    const long rows_k = varlen ? (long)Lk : (long)B * Lk;
    const size_t n_sem = (size_t)bwd_semaphore_count(B, H, Lq, varlen);
    const int split = bwd_head_split(B, Hkv, H / Hkv, Lk, varlen);
    w.dq_off = 0;
    w.delta_off = align256(rows_q * H * d * sizeof(float));
    w.part_off = w.delta_off + align256(rows_q * H * sizeof(float));
    w.sem_off = w.part_off + align256(bwd_partial_bytes(split, rows_k, Hkv, d, dv));
    w.total = w.sem_off + align256(n_sem * sizeof(int)) + align256(sizeof(VarlenMap));
    return w;
}

}  // namespace

extern "C" size_t attn_bwd_ex_workspace_size(int B, int H, int Hkv, int Lq, int Lk, int d, int d_v, int causal,
                                             int deterministic) {
    (void)causal;
    (void)deterministic;
    if (B < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || Lq < 0 || Lk < 0 || d <= 0 || d_v <= 0) return 0;
    // varlen and dense share the formula when Lq and Lk are the packed count;
    // the varlen semaphore bound is the larger one, so take the maximum.
    BwdWorkspace a = bwd_layout(B, H, Hkv, Lq, Lk, d, d_v, false), b = bwd_layout(B, H, Hkv, Lq, Lk, d, d_v, true);
    return a.total > b.total ? a.total : b.total;
}

extern "C" size_t attn_bwd_gqa_workspace_size(int B, int H, int Hkv, int Lq, int Lk, int d, int causal,
                                              int deterministic) {
    return attn_bwd_ex_workspace_size(B, H, Hkv, Lq, Lk, d, d, causal, deterministic);
}

extern "C" size_t attn_bwd_workspace_size(int B, int H, int Lq, int Lk, int d, int causal, int deterministic) {
    return attn_bwd_gqa_workspace_size(B, H, H, Lq, Lk, d, causal, deterministic);
}

namespace {

// The backward behind every entry point (cu_seqlens_k as in fwd_entry).
int bwd_entry(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
              void* dq, void* dk, void* dv, int B, int H, int Hkv, int Lq, int Lk, int d, int d_v, float scale,
              int causal, int window_left, int window_right, const unsigned char* block_mask, int mask_heads,
              const int* cu_seqlens, const int* cu_seqlens_k, int deterministic, void* workspace, size_t ws_bytes,
              cudaStream_t stream) {
    int rc = check_common(B, H, Lq, Lk, d, scale, cu_seqlens, cu_seqlens_k);
    if (rc) return rc;
    rc = check_block_mask(block_mask, mask_heads, H, cu_seqlens);
    if (rc) return rc;
    rc = check_window(window_left, window_right);
    if (rc) return rc;
    rc = check_heads(H, Hkv);
    if (rc) return rc;
    if (d_v != d && !(d == 192 && d_v == 128))
        return fail(ATTN_ERR_ARG, "head dims d=%d, d_v=%d not supported (d_v = d, or d = 192 with d_v = 128)", d,
                    d_v);
    const bool varlen = cu_seqlens != nullptr;
    const long rows_q = varlen ? (long)Lq : (long)B * Lq;
    const long rows_k = varlen ? (long)Lk : (long)B * Lk;
    if (rows_q == 0 && rows_k == 0) return ok();   // nothing to compute; pointers may be null
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
        return fail(ATTN_ERR_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(ATTN_ERR_ALIGN, "tensor pointers must be 16-byte aligned");
    const size_t need = attn_bwd_ex_workspace_size(B, H, Hkv, Lq, Lk, d, d_v, causal, deterministic);
    if (!workspace || ws_bytes < need)
        return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ATTN_ERR_ALIGN, "workspace must be 256-byte aligned");
    DevInfo di;
    if (!device_info(&di)) return fail(ATTN_ERR_LAUNCH, "cannot query the current device");
    BwdWorkspace wl = bwd_layout(B, H, Hkv, Lq, Lk, d, d_v, varlen);
    char* ws = static_cast<char*>(workspace);
    BwdParams p{};
    p.g.B = B;
    p.g.H = H;
    p.g.Lq = Lq;
    p.g.Lk = Lk;
    p.g.d = d;
    p.g.Hkv = Hkv;
    p.g.group = H / Hkv;
    p.g.cu_seqlens = cu_seqlens;
    p.g.cu_seqlens_k = cu_seqlens ? cu_seqlens_k : nullptr;
    set_mask(&p.g, causal, window_left, window_right);
    p.g.scale = scale;
    p.g.scale_log2 = scale * kLog2e;
    p.mask.ptr = block_mask;
    p.mask.heads = mask_heads;
    p.o = static_cast<const __nv_bfloat16*>(o);
    p.dout = static_cast<const __nv_bfloat16*>(dout);
    p.lse = lse;
    p.dq_acc = reinterpret_cast<float*>(ws + wl.dq_off);
    p.delta = reinterpret_cast<float*>(ws + wl.delta_off);
    p.semaphores = reinterpret_cast<int*>(ws + wl.sem_off);
    p.dq = static_cast<__nv_bfloat16*>(dq);
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.deterministic = deterministic ? 1 : 0;
    p.nm = (Lk + 127) / 128;
    p.nq = (Lq + 127) / 128;
    // a work tile is one key block of one key/value head; it streams Q and dO
    // of the query heads of the group (of its share of them when split)
    p.split = bwd_head_split(B, Hkv, p.g.group, Lk, varlen);
    p.d_v = d_v;
    p.dkv_part = p.split > 1 ? reinterpret_cast<float*>(ws + wl.part_off) : nullptr;
    p.n_tiles = varlen ? 0 : B * Hkv * p.nm * p.split;
    p.head_section = head_section(Hkv, (varlen ? (rows_q / B) : Lq) * (long)p.g.group, d);
    p.status = di.status;
    p.wait_budget_ns = wait_budget_ns();
    CUtensorMap tq, tk, tv, tdo, tdq;
    PairMaps pm = {};
    const bool pairs = g_bwd_pairs.load() != 0;
    const long qrows = rows_q > 0 ? rows_q : rows_k;
    const long krows = rows_k > 0 ? rows_k : rows_q;
    // Without query rows (or keys) the matching descriptors are never used; they
    // view the other tensor, with the heads of the smaller one so they stay in bounds.
    const int hq_map = rows_q > 0 ? H : Hkv;
    const void* qsrc = rows_q > 0 ? q : k;
    const void* dosrc = rows_q > 0 ? dout : k;
    // (v and dO are d_v <= d wide, so a fallback view of q or k with that width stays in bounds too)
    if (!make_map(&tq, qsrc, qrows, hq_map, d) || !make_map(&tk, rows_k > 0 ? k : q, krows, Hkv, d) ||
        !make_map(&tv, rows_k > 0 ? v : q, krows, Hkv, d_v) || !make_map(&tdo, dosrc, qrows, hq_map, d_v) ||
        !make_map_f32(&tdq, p.dq_acc, qrows, hq_map, d) || !make_map(&pm.q64, qsrc, qrows, hq_map, d, 64) ||
        !make_map(&pm.do64, dosrc, qrows, hq_map, d_v, 64) || !make_map_f32(&pm.dq32, p.dq_acc, qrows, hq_map, d, 32))
        return fail(ATTN_ERR_LAUNCH, "cuTensorMapEncodeTiled failed");
    // the pair backward's 32-column halves at head dim 64
    if (pairs && d == 64 && d_v == 64 &&
        (!make_map(&pm.q32, qsrc, qrows, hq_map, d, 128, true) || !make_map(&pm.do32, dosrc, qrows, hq_map, d, 128, true) ||
         !make_map(&pm.k32, rows_k > 0 ? k : q, krows, Hkv, d, 128, true)))
        return fail(ATTN_ERR_LAUNCH, "cuTensorMapEncodeTiled failed");
    cudaError_t e = launch_bwd(tq, tk, tv, tdo, tdq, pm, pairs, p, di.sms, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "backward launch failed: %s", cudaGetErrorString(e));
    return ok();
}

}  // namespace

extern "C" int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Lq, int Lk,
                            int d, float scale, int causal, const int* cu_seqlens, int deterministic,
                            void* workspace, size_t ws_bytes, cudaStream_t stream) {
    return bwd_entry(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Lq, Lk, d, d, scale, causal, -1, -1, nullptr, 1,
                     cu_seqlens, cu_seqlens, deterministic, workspace, ws_bytes, stream);
}

extern "C" int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                           const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Lq, int Lk,
                           int d, int d_v, float scale, int causal, int window_left, int window_right,
                           const unsigned char* block_mask, int mask_heads, const int* cu_seqlens_q,
                           const int* cu_seqlens_k, int deterministic, void* workspace, size_t ws_bytes,
                           cudaStream_t stream) {
    if (cu_seqlens_k && !cu_seqlens_q) return fail(ATTN_ERR_ARG, "attn_bwd_ex: key offsets without query offsets");
    return bwd_entry(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Lq, Lk, d, d_v, scale, causal, window_left,
                     window_right, block_mask, mask_heads, cu_seqlens_q, cu_seqlens_k ? cu_seqlens_k : cu_seqlens_q,
                     deterministic, workspace, ws_bytes, stream);
}

extern "C" int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Tq,
                               int Tk, int d, float scale, int causal, const int* cu_seqlens_q,
                               const int* cu_seqlens_k, int deterministic, void* workspace, size_t ws_bytes,
                               cudaStream_t stream) {
    if (!cu_seqlens_q || !cu_seqlens_k) return fail(ATTN_ERR_ARG, "attn_bwd_varlen: null offsets");
    return bwd_entry(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Tq, Tk, d, d, scale, causal, -1, -1, nullptr, 1,
                     cu_seqlens_q, cu_seqlens_k, deterministic, workspace, ws_bytes, stream);
}

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int d,
                        float scale, int causal, const int* cu_seqlens, int deterministic, void* workspace,
                        size_t ws_bytes, cudaStream_t stream) {
    return attn_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, B, H, H, Lq, Lk, d, scale, causal, cu_seqlens,
                        deterministic, workspace, ws_bytes, stream);
}

// ---------------------------------------------------------------- backward without allocation
// Scratch memory for attn_bwd_noalloc: the fp32 dQ accumulator, the D_i terms,
// the semaphores and the varlen map of one backward call. It lives in a
// file-scope device array, so every GPU that loads this library holds it
// until the process exits, and every call on a device shares it.
namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

// Device address of g_bwd_scratch on the current device, looked up once per
// device. The name g_bwd_scratch in host code is only a host-side stand-in,
// never a device address, so the address must come from the runtime.
bool scratch_address(void** out, cudaError_t* err) {
    static std::mutex mu;
    static void* cache[64] = {};
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return false;
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_bwd_scratch);
        if (*err != cudaSuccess) return false;
        cache[dev] = p;
    }
    *out = cache[dev];
    return true;
}

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                const void* dout, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk,
                                int d, float scale, int causal, const int* cu_seqlens, int deterministic,
                                cudaStream_t stream) {
    const size_t need = attn_bwd_workspace_size(B, H, Lq, Lk, d, causal, deterministic);
    if (need > (size_t)ATTN_NOALLOC_SCRATCH_BYTES)
        return fail(ATTN_ERR_WORKSPACE,
                    "attn_bwd_noalloc: this problem needs %zu bytes of scratch but the built-in array holds %zu; "
                    "call attn_bwd with a workspace instead",
                    need, (size_t)ATTN_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    cudaError_t e = cudaSuccess;
    if (!scratch_address(&scratch, &e))
        return fail(ATTN_ERR_LAUNCH, "attn_bwd_noalloc: cannot get the scratch array's device address: %s",
                    cudaGetErrorString(e));
    // the backward's preprocess kernel zeroes the accumulator and the semaphores on every call
    return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Lq, Lk, d, scale, causal, cu_seqlens, deterministic,
                    scratch, (size_t)ATTN_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" int attn_set_backward_cta_pairs(int enable) { return g_bwd_pairs.exchange(enable ? 1 : 0); }

extern "C" int attn_set_exp2_emulation(int d, int every) {
    if (d != 64 && d != 128) return fail(ATTN_ERR_ARG, "exp2 emulation applies to head dims 64 and 128, not %d", d);
    if (every != 0 && every != 4 && every != 8)
        return fail(ATTN_ERR_ARG, "exp2 emulation: one pair in 0 (off), 4 or 8, not %d", every);
    return g_poly_every[d == 64 ? 0 : 1].exchange(every);
}

extern "C" const char* attn_last_error(void) { return g_err; }

extern "C" int attn_check_status(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "stream error: %s", cudaGetErrorString(e));
    int st = 0;
    e = cudaMemcpyFromSymbol(&st, g_attn_status, sizeof(int));
    if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "cannot read the status word: %s", cudaGetErrorString(e));
    if (st != kStatusOk) {
        int zero = 0;
        cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int));
        if (st == kStatusMisaligned)
            return fail(ATTN_ERR_LAUNCH, "dynamic shared memory was not 1024-byte aligned");
        return fail(ATTN_ERR_TIMEOUT, "a kernel gave up waiting (status %d)", st);
    }
    return ok();
}

extern "C" int attn_version(void) { return 100; }
