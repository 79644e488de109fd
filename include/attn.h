/*
 * attn.h -- C ABI of libattn.so: exact multi-head scaled-dot-product attention
 * (forward and backward) on one NVIDIA GB300 GPU (sm_103a).
 *
 * The operation (FlashAttention-4 paper: Abstract and Section 1 -- exact
 * attention; Section 2.1 "Multi-head attention", empty in the page, read as the
 * textbook definition; Section 3.2.2 -- the five backward products). For each
 * batch entry b and head h, with s_ij = scale * <q_i, k_j>:
 *
 *   allowed(i, j) = j < Lk                     (causal == 0)
 *                 = j <= i + (Lk - Lq)         (causal != 0, bottom-right aligned)
 *   LSE_i = ln sum_{allowed j} exp(s_ij)        (natural log; -inf if no j allowed)
 *   O_i   = sum_j exp(s_ij - LSE_i) v_j         (0 if no j allowed)
 *   with loss L = sum(O * dO):
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i,
 *   dS_ij = P_ij (<dO_i, v_j> - <dO_i, O_i>),   P_ij = exp(s_ij - LSE_i).
 *
 * Layouts (row-major, contiguous, element types given):
 *   dense  (cu_seqlens == NULL): q, o, dq, dO  bf16 [B, Lq, H, d];
 *                                k, v, dk, dv  bf16 [B, Lk, H, d];
 *                                lse           fp32 [B, H, Lq].
 *   varlen (cu_seqlens != NULL): B sequences packed back to back; Lq and Lk
 *          are BOTH the packed row count T (they must be equal: one
 *          cu_seqlens serves queries and keys); cu_seqlens is a DEVICE int32
 *          array of B+1 nondecreasing offsets with cu_seqlens[0] = 0 and
 *          cu_seqlens[B] = T; tensors are [T, H, d], lse is fp32 [H, T].
 *          Sequence b covers rows cu_seqlens[b] .. cu_seqlens[b+1]-1 and attends
 *          only within itself. 1 <= B <= 1024.
 *   varlen with key offsets of their own (attn_fwd_varlen, attn_bwd_varlen):
 *          cu_seqlens_q packs the queries (Tq rows) and cu_seqlens_k the keys
 *          (Tk rows) of the same B sequences; sequence b has Lq_b =
 *          cu_seqlens_q[b+1]-cu_seqlens_q[b] queries and Lk_b keys and is
 *          its own rectangular problem, causal bottom-right aligned within it
 *          (j <= i + Lk_b - Lq_b); q, o, dq, dO are [Tq, H, d], k, v, dk, dv
 *          [Tk, Hkv, d], lse fp32 [H, Tq]. Either length may be 0 for a
 *          sequence (no keys: O = 0, LSE = -inf). Both arrays on the device,
 *          same rules as cu_seqlens.
 *   local window (attn_fwd_ex, attn_bwd_ex): window_left >= 0 drops keys
 *          j < i + (Lk - Lq) - window_left, window_right >= 0 keys
 *          j > i + (Lk - Lq) + window_right (per sequence for varlen); -1
 *          leaves that side open; causal != 0 sets window_right = 0. A row
 *          with no key left gets O = 0, LSE = -inf. The causal mask is the
 *          band (-1, 0). (FlashAttention-4 paper, Section 4: masking
 *          strategies compose with varlen and scheduling.)
 *   block mask (attn_fwd_ex, attn_bwd_ex; dense problems only): a DEVICE
 *          byte array [mask_heads][ceil(Lq/128)][ceil(Lk/128)], mask_heads 1
 *          (one mask for every head) or H (query head h uses its own); a zero
 *          byte drops all pairs of that 128-query x 128-key block, on top of
 *          the causal or window mask (FlashAttention-4 paper, Section 4:
 *          block-sparse patterns). Work tiles skip dropped blocks.
 *   grouped heads (attn_fwd_gqa, attn_bwd_gqa): k, v, dk, dv have Hkv heads
 *          instead of H ([B, Lk, Hkv, d] or [T, Hkv, d]); H must be a
 *          multiple of Hkv, and query head h reads key/value head
 *          h / (H / Hkv), so consecutive query heads share one (multi-query
 *          attention: Hkv = 1). dk and dv of a key/value head sum over the
 *          query heads that read it. The other entry points are Hkv = H.
 *
 * Arguments common to all calls:
 *   d       head dimension: 64, 128, 192 or 256 (forward and backward).
 *   scale   softmax scale, finite and > 0 (typically 1/sqrt(d)).
 *   causal  0 or 1.
 *   stream  CUDA stream the work is enqueued on; calls are asynchronous and
 *           never synchronise the host (except attn_check_status).
 *
 * Ownership: every pointer is caller-owned device memory, 16-byte aligned.
 * The library allocates no device memory; the backward pass takes a caller-
 * provided workspace. Inputs are read-only; outputs are fully overwritten.
 *
 * Errors: 0 on success, else a negative code; attn_last_error() returns a
 * thread-local message describing the last failure on the calling thread.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_OK 0
#define ATTN_ERR_ARG (-1)          /* null pointer, unsupported d, bad sizes or scale */
#define ATTN_ERR_ALIGN (-2)        /* a pointer is not 16-byte aligned */
#define ATTN_ERR_LAUNCH (-3)       /* a CUDA call or kernel launch failed */
#define ATTN_ERR_WORKSPACE (-4)    /* workspace missing or too small */
#define ATTN_ERR_TIMEOUT (-5)      /* a kernel gave up waiting (reported by attn_check_status) */

/*
 * Forward pass: writes o and lse (see the definitions above).
 * Tiles of 2x128 query rows (d <= 128; one 128-row tile for d = 192, 256)
 * run on a persistent grid (one CTA per SM) in a longest-first order
 * (FlashAttention-4 paper, Section 3.3 "Scheduling"); varlen batches are
 * sorted longest-first on the device.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int Lq, int Lk, int d, float scale, int causal,
             const int* cu_seqlens, cudaStream_t stream);

/*
 * Forward pass with a head dim of its own for v and o: q and k are
 * [.., H, d], v and o are [.., H, dv] (o has the rows of q). Supported:
 * dv = d (the same as attn_fwd), and d = 192 with dv = 128 (the shape of the
 * FlashAttention-4 paper's Section 5.1, Fig. 5). LSE as in attn_fwd. Other
 * pairs return ATTN_ERR_ARG. The backward for dv != d is attn_bwd_ex.
 */
int attn_fwd_hdim(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int H, int Lq, int Lk, int d, int dv, float scale, int causal,
                  const int* cu_seqlens, cudaStream_t stream);

/*
 * Forward pass with grouped key/value heads (see "grouped heads" above) and a
 * head dim of its own for v and o (the pairs attn_fwd_hdim accepts). The
 * query heads of a group are walked next to one another, so the group's K and
 * V are read from L2 after their first load (FlashAttention-4 paper,
 * Section 3.3, MQA/GQA order). Hkv < 1 or H not a multiple of Hkv returns
 * ATTN_ERR_ARG.
 */
int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int Hkv, int Lq, int Lk, int d, int dv, float scale, int causal,
                 const int* cu_seqlens, cudaStream_t stream);

/*
 * Bytes of device workspace attn_bwd needs for this problem (same size
 * arguments as attn_bwd; for varlen pass Lq = Lk = T). The workspace holds the
 * fp32 dQ accumulator, the row terms D_i = <dO_i, O_i>, and the semaphores of
 * the deterministic mode. Its contents need not be initialised.
 */
size_t attn_bwd_workspace_size(int B, int H, int Lq, int Lk, int d, int causal, int deterministic);

/*
 * Backward pass: given q, k, v, the forward's o and lse, and dO, writes dq,
 * dk, dv (bf16, layouts of q, k, v). FlashAttention-4 paper, Section 3.2:
 * the kernel iterates over K/V blocks, recomputes S^T, keeps P^T and the
 * dK/dV accumulators in tensor memory, and accumulates dQ with fp32 global
 * atomics (Section 3.2.2); for d = 192 and 256 each K/V block is worked on
 * in two 128-column chunks of dK/dV/dQ, each recomputing S^T and dP^T, so
 * that the accumulators fit in tensor memory. deterministic != 0 serialises
 * each dQ tile's accumulation in a fixed order with semaphores so repeated
 * calls are bit-identical (Section 3.2.4). workspace/ws_bytes: caller-owned device
 * memory of at least attn_bwd_workspace_size(...) bytes, 256-byte aligned,
 * not used concurrently by another call.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv,
             int B, int H, int Lq, int Lk, int d, float scale, int causal,
             const int* cu_seqlens, int deterministic, void* workspace, size_t ws_bytes,
             cudaStream_t stream);

/*
 * Forward pass of a packed batch whose sequences have key lengths of their
 * own (see "varlen with key offsets" above), e.g. prefill and decode steps
 * in one call (FlashAttention-4 paper, Section 3.3, varlen scheduling).
 * Grouped heads and the head-dim pairs as in attn_fwd_gqa. Sequences are
 * walked longest first by key count (the longest work tile of a sequence
 * visits all its keys). Null offsets return ATTN_ERR_ARG.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int Hkv, int Tq, int Tk, int d, int dv, float scale, int causal,
                    const int* cu_seqlens_q, const int* cu_seqlens_k, cudaStream_t stream);

/*
 * The general forward: every entry point above is this one with some
 * arguments fixed. Hkv key/value heads (grouped heads), a head dim d_v of
 * its own for v and o (d_v = d, or d = 192 with d_v = 128), a local window
 * (window_left, window_right; -1, -1 for none; see above), a block mask
 * (block_mask, mask_heads; NULL for none; see above), and either
 * dense tensors (cu_seqlens_q == NULL, cu_seqlens_k == NULL), packed
 * sequences with one offset array (cu_seqlens_k == NULL: Lq = Lk = T), or
 * packed sequences with key offsets of their own (Lq = Tq, Lk = Tk).
 * cu_seqlens_k without cu_seqlens_q, a window bound below -1, or a block
 * mask with offsets or mask_heads not 1 or H, returns ATTN_ERR_ARG. The work tiles visit only the key blocks their rows' band
 * reaches.
 */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int Hkv, int Lq, int Lk, int d, int d_v, float scale, int causal,
                int window_left, int window_right, const unsigned char* block_mask, int mask_heads,
                const int* cu_seqlens_q, const int* cu_seqlens_k, cudaStream_t stream);

/*
 * Workspace for attn_bwd_ex (any of the arguments attn_bwd_ex accepts).
 */
size_t attn_bwd_ex_workspace_size(int B, int H, int Hkv, int Lq, int Lk, int d, int d_v, int causal,
                                  int deterministic);

/*
 * The general backward, arguments as in attn_fwd_ex (dv here is the dV
 * output; d_v the head dim of v, o, dO and dV). With d = 192 and d_v = 128
 * the d = 192 kernel's two column chunks split dK and dQ at column 128;
 * chunk 0 also owns all of dV and chunk 1 skips the dV product, and the
 * products with V and dO contract over their 128 columns.
 */
int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dout, void* dq, void* dk, void* dv,
                int B, int H, int Hkv, int Lq, int Lk, int d, int d_v, float scale, int causal,
                int window_left, int window_right, const unsigned char* block_mask, int mask_heads,
                const int* cu_seqlens_q, const int* cu_seqlens_k, int deterministic,
                void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * Workspace for attn_bwd_gqa: as attn_bwd_workspace_size, plus fp32 slots
 * for partial dK and dV when the backward splits a group's query heads over
 * several work tiles (see attn_bwd_gqa). Hkv = H gives attn_bwd_workspace_size.
 * Returns 0 for invalid sizes (including H not a multiple of Hkv).
 */
size_t attn_bwd_gqa_workspace_size(int B, int H, int Hkv, int Lq, int Lk, int d, int causal,
                                   int deterministic);

/*
 * Backward pass with grouped key/value heads (see "grouped heads" above; dv
 * = d). A work tile is one 128-key block of one key/value head: it visits the
 * query blocks of the group's query heads in turn and keeps their dK and dV
 * in tensor memory. When that gives fewer than 640 work tiles (about four per
 * SM, too few to balance causal work), the group's query heads are split
 * over the smallest number of tiles per key block (a divisor of H / Hkv) that
 * reaches 640; each writes partial dK and dV to fp32 workspace slots that a
 * last kernel sums in slot order. Either way dK and dV need no atomics and
 * are bit-identical across runs even with deterministic = 0 (the
 * FlashAttention-4 paper, Section 3.2.4, reduces them across CTAs with
 * atomics instead). workspace: attn_bwd_gqa_workspace_size(...) bytes.
 */
int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv,
                 int B, int H, int Hkv, int Lq, int Lk, int d, float scale, int causal,
                 const int* cu_seqlens, int deterministic, void* workspace, size_t ws_bytes,
                 cudaStream_t stream);

/*
 * Backward pass of a packed batch with key offsets of their own (dv = d);
 * otherwise as attn_bwd_gqa. Sequences are walked longest first by query
 * count (the backward's work tiles are key blocks, and the longest visits
 * every query block). workspace: attn_bwd_gqa_workspace_size(B, H, Hkv, Tq,
 * Tk, d, causal, deterministic) bytes.
 */
int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv,
                    int B, int H, int Hkv, int Tq, int Tk, int d, float scale, int causal,
                    const int* cu_seqlens_q, const int* cu_seqlens_k, int deterministic,
                    void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * Backward pass that allocates nothing: the same operation, arguments and
 * results as attn_bwd, minus the workspace. It is meant for callers that
 * cannot hand the library device memory of its own -- for instance code
 * running inside a host framework or serving runtime that owns the whole
 * device memory pool (allocations outside its planner are forbidden once it
 * runs), or a plugin that only receives the input and output pointers.
 * (The FlashAttention-4 paper has no counterpart to this entry point.)
 *
 * Its scratch memory is a fixed array of ATTN_NOALLOC_SCRATCH_BYTES inside
 * this library, which every GPU that loads the library holds until the
 * process exits. Problems whose attn_bwd_workspace_size(...) exceeds it are
 * rejected with ATTN_ERR_WORKSPACE (use attn_bwd with a workspace for them).
 * It calls no cudaMalloc/cudaFree and no allocating library routine.
 *
 * The first call on each device looks up the array's device address (set-up
 * done once per device, with that device current); make that first call
 * before any stream capture. All calls on a device share the one array and
 * it keeps the previous call's contents: each call clears what must start at
 * zero itself, but calls that overlap on the GPU (e.g. on two streams at
 * once) race on the array and must be serialised by the caller.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv,
                     int B, int H, int Lq, int Lk, int d, float scale, int causal,
                     const int* cu_seqlens, int deterministic, cudaStream_t stream);

/*
 * Partial emulation of the forward's exponentials (FlashAttention-4 paper,
 * Section 3.1.3, "partial emulation"; FA4 blog, "关键实现技术"): for head dim d
 * (64 or 128), `every` = 8 or 4 computes one score-column pair in every 8 or 4
 * (12.5% or 25% of the entries) with a degree-3 Cody-Waite + Horner polynomial
 * on the FMA pipes instead of the MUFU ex2 unit, except on each row's last K/V
 * block; 0 uses MUFU for all. Results differ from MUFU's by at most one bf16
 * ulp of P. It applies to the plain forward kernel (no left window bound, no
 * block mask). The setting is process-wide (all threads, all devices) and
 * takes effect at the next forward call; the default per head dim is the one
 * measured faster on GB300.
 * Returns the previous setting (>= 0), or ATTN_ERR_ARG for another d or
 * `every` value.
 */
int attn_set_exp2_emulation(int d, int every);

/*
 * Backward on CTA pairs (FlashAttention-4 paper, Section 3.2.3 "2-CTA backward
 * pass"; Section 2.2 "2-CTA tensor cores"): with `enable` != 0 the backward's
 * main kernel runs on clusters of two CTAs whose tensor cores work as one
 * (tcgen05 .cta_group::2): each pair owns 256 keys, the S^T, dP^T, dV and dK
 * products run with M = 256 and each CTA stages half of operand B, and dQ is
 * summed over the pair's 256 keys by the MMA itself, so each CTA adds a
 * 64-row dQ tile per query block (half the global reduce-adds of single
 * CTAs). It applies where supported: head dim 64 or 128, the same for q, k
 * and v, grouped heads or not, no window beyond the causal mask, no block mask (dense or
 * packed, deterministic or not); other problems run on single CTAs.
 * Results agree with the single-CTA kernels to rounding (the order of the fp32
 * sums differs); the deterministic mode stays bit-identical run to run. The
 * setting is process-wide and takes effect at the next backward call; the
 * default is the one measured faster on GB300.
 * Returns the previous setting (0 or 1).
 */
int attn_set_backward_cta_pairs(int enable);

/* Message for the last nonzero return code on this thread ("" if none). */
const char* attn_last_error(void);

/*
 * Synchronises `stream`, then reports (and clears) the device status word the
 * kernels set when a bounded wait ran out: 0 if clean, ATTN_ERR_TIMEOUT if a
 * kernel gave up, ATTN_ERR_LAUNCH if the stream reports a CUDA error.
 */
int attn_check_status(cudaStream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
