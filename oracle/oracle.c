/*
 * fp64 CPU oracle for exact multi-head scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do. It shares no code, header, table or helper with the CUDA
 * library, and it includes nothing from it.
 *
 * What it computes is the plain textbook definition (FlashAttention-4 paper,
 * "Abstract" and Section 1: the method is *exact* attention; Section 2.1
 * "Multi-head attention" is empty in the page, so the standard definition is
 * used). Per batch b and head h, with s_ij = scale * <q_i, k_j>:
 *
 *     allowed(i, j) = j < Lk                       (non-causal)
 *                   = j <= i + (Lk - Lq)           (causal, bottom-right aligned)
 *   and with a local window (window_left wl, window_right wr; -1: no bound;
 *   causal means wr = 0), with delta = Lk - Lq:
 *     allowed(i, j) = 0 <= j < Lk,  j >= i + delta - wl (wl >= 0),
 *                     j <= i + delta + wr (wr >= 0)
 *   (a band around the bottom-right diagonal: the FlashAttention-4 paper's
 *   Section 4 lists masking strategies among the primitives its kernels
 *   compose; the band is the plainest one beyond the causal mask),
 *   and with a block mask (dense problems; same section: block-sparse
 *   patterns are one of those primitives): a byte array
 *   block_mask[mask_heads][ceil(Lq / block_q)][ceil(Lk / block_k)], mask_heads
 *   1 (shared) or H (query head h uses its own); allowed(i, j) also needs
 *   block_mask[h or 0][i / block_q][j / block_k] != 0.
 *     LSE_i = m_i + ln sum_j exp(s_ij - m_i),  m_i = max_j s_ij   (allowed j)
 *     P_ij  = exp(s_ij - LSE_i)
 *     O_i   = sum_j P_ij v_j
 *
 * q and k have head dim d; v, o, dout and dv have their own head dim dv
 * (equal to d for the textbook case; the FlashAttention-4 paper's Section 5.1
 * also measures d = 192 for q/k with 128 for v, Fig. 5).
 *
 * Grouped heads (multi-query and grouped-query attention, which the paper's
 * Section 3.3 schedules by key/value head): q, o, dout, dq have H heads; k, v,
 * dk, dv have Hkv heads (H a multiple of Hkv), and query head h reads
 * key/value head h / (H / Hkv), so consecutive query heads share one key/value
 * head. dk and dv of a key/value head sum over the query heads of its group.
 * Hkv = H is the plain multi-head case.
 *
 * Backward, for the scalar loss L = sum(O * dO) (FlashAttention-4 paper,
 * Section 3.2.2: five products -- S recomputed, dP = dO V^T, dV = P^T dO,
 * dQ = dS K, dK = dS^T Q):
 *
 *     dP_ij = <dO_i, v_j>,   D_i = <dO_i, O_i>,   dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale * sum_j dS_ij k_j
 *     dK_j  = scale * sum_i dS_ij q_i
 *     dV_j  = sum_i P_ij dO_i
 *
 * A row with no allowed key (causal with Lq > Lk, or a window that holds no
 * key of the row) has
 * O_i = 0, LSE_i = -inf, and contributes nothing to any gradient.
 *
 * Every output element is evaluated directly from its formula, with a single
 * running accumulator per sum in index order; there is no blocking, tiling,
 * online softmax or reordering. Threads only split the set of independent
 * outputs (rows of O / dQ, rows of dK / dV) between them.
 *
 * Layouts (row-major, element counts):
 *   dense  : q, o, dq  [B, Lq, H, d];  k, v, dk, dv [B, Lk, Hkv, d];  lse [B, H, Lq]
 *   varlen : cu_seqlens[B+1] (host, int32) packs B sequences of queries;
 *            cu_seqlens_k[B+1] packs their keys (NULL: the same offsets, so
 *            Lk_b = Lq_b). Sequence b has Lq_b = cu[b+1]-cu[b] query rows
 *            and Lk_b = cu_k[b+1]-cu_k[b] keys, each its own problem (causal
 *            bottom-right aligned within it, as the FlashAttention-4 paper's
 *            Section 3.3 mixes sequences of different query and key lengths);
 *            q, o, dq [Tq, H, d]; k, v, dk, dv [Tk, Hkv, d]; lse [H, Tq]
 *            (Tq = cu[B], Tk = cu_k[B]); Lq and Lk are then ignored.
 *
 * Row subsets: `rows` (nrows entries) lists query-row indices, relative to
 * each sequence, whose O / LSE / dQ are wanted; `krows` lists key-row indices
 * whose dK / dV are wanted. NULL means every row. Entries out of range for a
 * sequence are skipped. Outputs outside the subset are left untouched.
 *
 * Return value: 0 on success, -1 on a bad argument, -2 on allocation failure.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *dout;
    double *o, *lse, *dq, *dk, *dv;
    int B, H, Hkv, Lq, Lk, d, dvh;   /* Hkv: heads of k, v; dvh: head dim of v, o, dout, dv */
    int wl, wr;                      /* window bounds (-1: none); causal is wr = 0 */
    const unsigned char *bmask;      /* block mask or NULL; heads bm_h, block sizes bm_q x bm_k */
    int bm_h, bm_q, bm_k;
    double scale;
    const int *cu;          /* NULL for dense */
    const int *cuk;         /* key offsets (varlen): cu_seqlens_k, or cu */
    /* per (b, h, row) statistics used by the backward pass */
    double *lse_all;        /* [B*H*Lq_max] or varlen [H*T] */
    double *D_all;
    /* work list */
    const int *items;       /* (b, h, row) triples, flattened */
    long n_items;
    atomic_long next;
    int phase;
} job_t;

/* ---- sequence geometry ------------------------------------------------- */

static int seq_lq(const job_t *J, int b) { return J->cu ? J->cu[b + 1] - J->cu[b] : J->Lq; }
static int seq_lk(const job_t *J, int b) { return J->cu ? J->cuk[b + 1] - J->cuk[b] : J->Lk; }

/* element offset of row i of sequence b, head h, in a [.., L, H, d] tensor */
static long row_off(const job_t *J, int b, int i, int h, int L) {
    if (J->cu) return ((long)(J->cu[b] + i) * J->H + h) * J->d;
    return (((long)b * L + i) * J->H + h) * J->d;
}

/* the same for a [.., L, H, dv] tensor (v, o, dout, dv) */
static long row_off_v(const job_t *J, int b, int i, int h, int L) {
    if (J->cu) return ((long)(J->cu[b] + i) * J->H + h) * J->dvh;
    return (((long)b * L + i) * J->H + h) * J->dvh;
}

/* key/value head read by query head h */
static int kvh(const job_t *J, int h) { return h / (J->H / J->Hkv); }

/* element offset of row j of key/value head hk in a [.., L, Hkv, d] tensor (k, dk) */
static long row_off_k(const job_t *J, int b, int j, int hk, int L) {
    if (J->cu) return ((long)(J->cuk[b] + j) * J->Hkv + hk) * J->d;
    return (((long)b * L + j) * J->Hkv + hk) * J->d;
}

/* the same with head dim dvh (v, dv) */
static long row_off_kv(const job_t *J, int b, int j, int hk, int L) {
    if (J->cu) return ((long)(J->cuk[b] + j) * J->Hkv + hk) * J->dvh;
    return (((long)b * L + j) * J->Hkv + hk) * J->dvh;
}

/* index of (b, h, i) into an lse-shaped array */
static long stat_off(const job_t *J, int b, int h, int i) {
    if (J->cu) return (long)h * J->cu[J->B] + J->cu[b] + i;
    return ((long)b * J->H + h) * J->Lq + i;
}

/* does query row i of query head h see key j (batch entry / sequence b) */
static int allowed(const job_t *J, int b, int h, int i, int j) {
    int lq = seq_lq(J, b), lk = seq_lk(J, b);
    int delta = lk - lq;
    if (j < 0 || j >= lk) return 0;
    if (J->wr >= 0 && j > i + delta + J->wr) return 0;
    if (J->wl >= 0 && j < i + delta - J->wl) return 0;
    if (J->bmask) {
        int rows = (lq + J->bm_q - 1) / J->bm_q, cols = (lk + J->bm_k - 1) / J->bm_k;
        int hm = J->bm_h == 1 ? 0 : h;
        if (!J->bmask[((long)hm * rows + i / J->bm_q) * cols + j / J->bm_k]) return 0;
    }
    return 1;
}

static double dot(const double *a, const double *b, int n) {
    double s = 0.0;
    for (int c = 0; c < n; c++) s += a[c] * b[c];
    return s;
}

static double score(const job_t *J, int b, int h, int i, int j) {
    const double *qi = J->q + row_off(J, b, i, h, J->Lq);
    const double *kj = J->k + row_off_k(J, b, j, kvh(J, h), J->Lk);
    return J->scale * dot(qi, kj, J->d);
}

/* LSE_i by the definition: max, then ln of the shifted sum of exponentials. */
static double row_lse(const job_t *J, int b, int h, int i) {
    int lk = seq_lk(J, b);
    double m = -INFINITY;
    for (int j = 0; j < lk; j++)
        if (allowed(J, b, h, i, j)) {
            double s = score(J, b, h, i, j);
            if (s > m) m = s;
        }
    if (m == -INFINITY) return -INFINITY;
    double sum = 0.0;
    for (int j = 0; j < lk; j++)
        if (allowed(J, b, h, i, j)) sum += exp(score(J, b, h, i, j) - m);
    return m + log(sum);
}

/* O_i = sum_j exp(s_ij - LSE_i) v_j  (written into out[0..dv)) */
static void row_out(const job_t *J, int b, int h, int i, double lse, double *out) {
    int dv = J->dvh, lk = seq_lk(J, b);
    for (int c = 0; c < dv; c++) out[c] = 0.0;
    if (lse == -INFINITY) return;
    for (int j = 0; j < lk; j++) {
        if (!allowed(J, b, h, i, j)) continue;
        double p = exp(score(J, b, h, i, j) - lse);
        const double *vj = J->v + row_off_kv(J, b, j, kvh(J, h), J->Lk);
        for (int c = 0; c < dv; c++) out[c] += p * vj[c];
    }
}

/* dS_ij = P_ij (<dO_i, v_j> - D_i) */
static double dscore(const job_t *J, int b, int h, int i, int j) {
    long st = stat_off(J, b, h, i);
    double p = exp(score(J, b, h, i, j) - J->lse_all[st]);
    const double *doi = J->dout + row_off_v(J, b, i, h, J->Lq);
    const double *vj = J->v + row_off_kv(J, b, j, kvh(J, h), J->Lk);
    return p * (dot(doi, vj, J->dvh) - J->D_all[st]);
}

/* ---- work items -------------------------------------------------------- */
/* items are (b, h, i) triples; the phase decides what is computed for them */

enum { PH_FWD = 0, PH_STATS = 1, PH_DQ = 2, PH_DKV = 3 };

static void do_item(job_t *J, int b, int h, int i) {
    int d = J->d, dv = J->dvh;
    if (J->phase == PH_FWD) {
        double lse = row_lse(J, b, h, i);
        J->lse[stat_off(J, b, h, i)] = lse;
        row_out(J, b, h, i, lse, J->o + row_off_v(J, b, i, h, J->Lq));
    } else if (J->phase == PH_STATS) {
        long st = stat_off(J, b, h, i);
        double *tmp = (double *)malloc(sizeof(double) * (size_t)dv);
        double lse = row_lse(J, b, h, i);
        row_out(J, b, h, i, lse, tmp);
        J->lse_all[st] = lse;
        J->D_all[st] = dot(J->dout + row_off_v(J, b, i, h, J->Lq), tmp, dv);
        free(tmp);
    } else if (J->phase == PH_DQ) {
        double *dqi = J->dq + row_off(J, b, i, h, J->Lq);
        int lk = seq_lk(J, b);
        for (int c = 0; c < d; c++) dqi[c] = 0.0;
        if (J->lse_all[stat_off(J, b, h, i)] == -INFINITY) return;
        for (int j = 0; j < lk; j++) {
            if (!allowed(J, b, h, i, j)) continue;
            double ds = dscore(J, b, h, i, j);
            const double *kj = J->k + row_off_k(J, b, j, kvh(J, h), J->Lk);
            for (int c = 0; c < d; c++) dqi[c] += ds * kj[c];
        }
        for (int c = 0; c < d; c++) dqi[c] *= J->scale;
    } else { /* PH_DKV: item (b, hk, j): key row j of key/value head hk, summed
                over the query heads of its group */
        int j = i, hk = h, lq = seq_lq(J, b), g = J->H / J->Hkv;
        double *dkj = J->dk + row_off_k(J, b, j, hk, J->Lk);
        double *dvj = J->dv + row_off_kv(J, b, j, hk, J->Lk);
        const double *vj = J->v + row_off_kv(J, b, j, hk, J->Lk);
        for (int c = 0; c < d; c++) dkj[c] = 0.0;
        for (int c = 0; c < dv; c++) dvj[c] = 0.0;
        for (int hq = hk * g; hq < hk * g + g; hq++)
            for (int r = 0; r < lq; r++) {
                if (!allowed(J, b, hq, r, j)) continue;
                long st = stat_off(J, b, hq, r);
                double p = exp(score(J, b, hq, r, j) - J->lse_all[st]);
                const double *dor = J->dout + row_off_v(J, b, r, hq, J->Lq);
                const double *qr = J->q + row_off(J, b, r, hq, J->Lq);
                double ds = p * (dot(dor, vj, dv) - J->D_all[st]);
                for (int c = 0; c < d; c++) dkj[c] += ds * qr[c];
                for (int c = 0; c < dv; c++) dvj[c] += p * dor[c];
            }
        for (int c = 0; c < d; c++) dkj[c] *= J->scale;
    }
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    for (;;) {
        long t = atomic_fetch_add(&J->next, 1);
        if (t >= J->n_items) break;
        const int *it = J->items + 3 * t;
        do_item(J, it[0], it[1], it[2]);
    }
    return NULL;
}

static void run_items(job_t *J, int phase, const int *items, long n, int nthreads) {
    J->phase = phase;
    J->items = items;
    J->n_items = n;
    atomic_store(&J->next, 0);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads == 1 || n < 2) { worker(J); return; }
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < nthreads; t++)
        if (pthread_create(&th[t], NULL, worker, J) == 0) started++;
        else break;
    if (started == 0) worker(J);
    for (int t = 0; t < started; t++) pthread_join(th[t], NULL);
}

/* Build the (b, h, i) list for a row subset; kind 0 = query rows, 1 = key rows. */
static int *make_items(const job_t *J, const int *rows, int nrows, int kind, long *n_out) {
    long cap = 0;
    for (int b = 0; b < J->B; b++) {
        int L = kind ? seq_lk(J, b) : seq_lq(J, b);
        cap += (long)(kind ? J->Hkv : J->H) * (rows ? nrows : L);
    }
    int *items = (int *)malloc(sizeof(int) * 3 * (size_t)(cap > 0 ? cap : 1));
    if (!items) return NULL;
    long n = 0;
    for (int b = 0; b < J->B; b++) {
        int L = kind ? seq_lk(J, b) : seq_lq(J, b);
        int cnt = rows ? nrows : L;
        for (int h = 0; h < (kind ? J->Hkv : J->H); h++)   /* key rows: key/value heads */
            for (int t = 0; t < cnt; t++) {
                int i = rows ? rows[t] : t;
                if (i < 0 || i >= L) continue;
                items[3 * n] = b; items[3 * n + 1] = h; items[3 * n + 2] = i;
                n++;
            }
    }
    *n_out = n;
    return items;
}

static int check_offsets(int B, const int *cu) {
    if (cu[0] != 0) return -1;
    for (int b = 0; b < B; b++) if (cu[b + 1] < cu[b]) return -1;
    return 0;
}

static int check_args(int B, int H, int Hkv, int Lq, int Lk, int d, int dv, const int *cu, const int *cuk,
                      int wl, int wr, const unsigned char *bmask, int bm_h, int bm_q, int bm_k) {
    if (B < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || d < 1 || dv < 1) return -1;
    if (wl < -1 || wr < -1) return -1;
    if (bmask && (cu || (bm_h != 1 && bm_h != H) || bm_q < 1 || bm_k < 1)) return -1;
    if (!cu && (Lq < 0 || Lk < 0)) return -1;
    if (cuk && !cu) return -1;
    if (cu && check_offsets(B, cu)) return -1;
    if (cuk && check_offsets(B, cuk)) return -1;
    return 0;
}

static void init_job(job_t *J, const double *q, const double *k, const double *v, const double *dout,
                     int B, int H, int Hkv, int Lq, int Lk, int d, int dv, double scale, int causal,
                     int wl, int wr, const int *cu, const int *cuk, const unsigned char *bmask, int bm_h,
                     int bm_q, int bm_k) {
    memset(J, 0, sizeof(*J));
    J->bmask = bmask; J->bm_h = bm_h; J->bm_q = bm_q; J->bm_k = bm_k;
    J->q = q; J->k = k; J->v = v; J->dout = dout;
    J->B = B; J->H = H; J->Hkv = Hkv; J->Lq = Lq; J->Lk = Lk; J->d = d; J->dvh = dv;
    J->scale = scale; J->wl = wl; J->wr = causal ? 0 : wr;
    J->cu = cu; J->cuk = cuk ? cuk : cu;
}

int oracle_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
               int B, int H, int Hkv, int Lq, int Lk, int d, int dv, double scale, int causal,
               int window_left, int window_right, const unsigned char *block_mask, int mask_heads,
               int block_q, int block_k,
               const int *cu_seqlens, const int *cu_seqlens_k, const int *rows, int nrows, int nthreads) {
    if (!q || !k || !v || !o || !lse) return -1;
    if (check_args(B, H, Hkv, Lq, Lk, d, dv, cu_seqlens, cu_seqlens_k, window_left, window_right, block_mask,
                   mask_heads, block_q, block_k)) return -1;
    job_t J;
    init_job(&J, q, k, v, NULL, B, H, Hkv, Lq, Lk, d, dv, scale, causal, window_left, window_right, cu_seqlens,
             cu_seqlens_k, block_mask, mask_heads, block_q, block_k);
    J.o = o; J.lse = lse;
    long n;
    int *items = make_items(&J, rows, nrows, 0, &n);
    if (!items) return -2;
    run_items(&J, PH_FWD, items, n, nthreads);
    free(items);
    return 0;
}

int oracle_bwd(const double *q, const double *k, const double *v, const double *dout,
               double *dq, double *dk, double *dv,
               int B, int H, int Hkv, int Lq, int Lk, int d, int dvd, double scale, int causal,
               int window_left, int window_right, const unsigned char *block_mask, int mask_heads,
               int block_q, int block_k,
               const int *cu_seqlens, const int *cu_seqlens_k, const int *qrows, int nqrows,
               const int *krows, int nkrows, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return -1;
    if (check_args(B, H, Hkv, Lq, Lk, d, dvd, cu_seqlens, cu_seqlens_k, window_left, window_right, block_mask,
                   mask_heads, block_q, block_k)) return -1;
    if ((qrows && nqrows < 0) || (krows && nkrows < 0)) return -1;
    job_t J;
    init_job(&J, q, k, v, dout, B, H, Hkv, Lq, Lk, d, dvd, scale, causal, window_left, window_right, cu_seqlens,
             cu_seqlens_k, block_mask, mask_heads, block_q, block_k);
    J.dq = dq; J.dk = dk; J.dv = dv;

    /* longest sequence, the range of relative row indices */
    int lmax = cu_seqlens ? 0 : Lq;
    if (cu_seqlens)
        for (int b = 0; b < B; b++) if (cu_seqlens[b + 1] - cu_seqlens[b] > lmax) lmax = cu_seqlens[b + 1] - cu_seqlens[b];
    long nstat = cu_seqlens ? (long)H * cu_seqlens[B] : (long)B * H * Lq;
    J.lse_all = (double *)malloc(sizeof(double) * (size_t)(nstat > 0 ? nstat : 1));
    J.D_all = (double *)malloc(sizeof(double) * (size_t)(nstat > 0 ? nstat : 1));
    unsigned char *need = (unsigned char *)calloc((size_t)(lmax > 0 ? lmax : 1), 1);
    int *list = (int *)malloc(sizeof(int) * (size_t)(lmax > 0 ? lmax : 1));
    if (!J.lse_all || !J.D_all || !need || !list) {
        free(J.lse_all); free(J.D_all); free(need); free(list);
        return -2;
    }

    /* Query rows whose LSE_i and D_i are needed: the requested dQ rows, plus
       every row that can see a requested key row (for a dense problem with a
       right bound wr, key j is seen by rows i >= j - (Lk - Lq) - wr only;
       otherwise by all rows). */
    int want_dq = !(qrows && nqrows == 0);
    int want_dkv = !(krows && nkrows == 0);
    if (want_dq) {
        if (!qrows) memset(need, 1, (size_t)lmax);
        else for (int t = 0; t < nqrows; t++) if (qrows[t] >= 0 && qrows[t] < lmax) need[qrows[t]] = 1;
    }
    if (want_dkv) {
        int i0 = 0;
        if (krows && J.wr >= 0 && !cu_seqlens) {
            int jmin = Lk;
            for (int t = 0; t < nkrows; t++) if (krows[t] >= 0 && krows[t] < jmin) jmin = krows[t];
            i0 = jmin - (Lk - Lq) - J.wr;
            if (i0 < 0) i0 = 0;
        }
        for (int i = i0; i < lmax; i++) need[i] = 1;
    }
    int nlist = 0;
    for (int i = 0; i < lmax; i++) if (need[i]) list[nlist++] = i;

    long n;
    int rc = 0;
    int *items = make_items(&J, list, nlist, 0, &n);
    if (!items) { rc = -2; goto done; }
    run_items(&J, PH_STATS, items, n, nthreads);
    free(items);

    if (want_dq) {
        items = make_items(&J, qrows, nqrows, 0, &n);
        if (!items) { rc = -2; goto done; }
        run_items(&J, PH_DQ, items, n, nthreads);
        free(items);
    }
    if (want_dkv) {
        items = make_items(&J, krows, nkrows, 1, &n);
        if (!items) { rc = -2; goto done; }
        run_items(&J, PH_DKV, items, n, nthreads);
        free(items);
    }
done:
    free(J.lse_all); free(J.D_all); free(need); free(list);
    return rc;
}
