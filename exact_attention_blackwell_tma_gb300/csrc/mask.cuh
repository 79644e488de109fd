// The attention mask as index arithmetic: which keys a query row sees and
// which query rows see a key, for the no-mask, causal and local-window cases.
//
// Query i of a sequence with lq queries and lk keys sees key j when
//   0 <= j < lk,  j <= i + delta + wr (wr >= 0),  j >= i + delta - wl (wl >= 0),
// delta = lk - lq (bottom-right aligned); wl / wr = -1: no bound on that side;
// causal is wr = 0. FlashAttention-4 paper, Section 4: masking strategies are
// one of the primitives its kernels compose with varlen and scheduling; the
// band is the plainest one beyond the causal mask and contains it.
//
// The functions are also compiled for the host, where tests/sched_host.cu
// checks them against a brute-force scan of the mask.
#pragma once

struct MaskBand {
    int delta;   // lk - lq
    int wl, wr;  // -1: no bound
    int lq, lk;
};

__host__ __device__ __forceinline__ MaskBand mask_band(int lq, int lk, int wl, int wr) {
    return MaskBand{lk - lq, wl, wr, lq, lk};
}

// Keys [lo, hi) that row r sees (hi <= lo: none).
__host__ __device__ __forceinline__ int band_key_lo(const MaskBand& m, int r) {
    const int lo = m.wl >= 0 ? r + m.delta - m.wl : 0;
    return lo > 0 ? lo : 0;
}
__host__ __device__ __forceinline__ int band_key_hi(const MaskBand& m, int r) {
    const int hi = m.wr >= 0 ? r + m.delta + m.wr + 1 : m.lk;
    return hi < m.lk ? hi : m.lk;
}

// Blocks of `bn` keys that rows r0..r1 (clamped to the sequence) see between
// them: [*jlo, *jhi). Returns false (and an empty range) if none. The rows'
// key ranges overlap or touch (consecutive rows shift the band by one key), so
// their union is one range.
__host__ __device__ __forceinline__ bool band_key_blocks(const MaskBand& m, int r0, int r1, int bn, int* jlo,
                                                         int* jhi) {
    if (r1 > m.lq - 1) r1 = m.lq - 1;
    if (r0 < 0) r0 = 0;
    *jlo = *jhi = 0;
    if (r0 > r1) return false;
    const int lo = band_key_lo(m, r0), hi = band_key_hi(m, r1);
    if (hi <= lo) return false;
    *jlo = lo / bn;
    *jhi = (hi + bn - 1) / bn;
    return true;
}

// Query rows [lo, hi) that see key j.
__host__ __device__ __forceinline__ int band_query_lo(const MaskBand& m, int j) {
    const int lo = m.wr >= 0 ? j - m.delta - m.wr : 0;
    return lo > 0 ? lo : 0;
}
__host__ __device__ __forceinline__ int band_query_hi(const MaskBand& m, int j) {
    const int hi = m.wl >= 0 ? j - m.delta + m.wl + 1 : m.lq;
    return hi < m.lq ? hi : m.lq;
}

// Blocks of `bm` query rows that see some key of keys k0..k1 (clamped to the
// sequence): [*mlo, *mhi). Returns false (and an empty range) if none.
__host__ __device__ __forceinline__ bool band_query_blocks(const MaskBand& m, int k0, int k1, int bm, int* mlo,
                                                           int* mhi) {
    if (k1 > m.lk - 1) k1 = m.lk - 1;
    if (k0 < 0) k0 = 0;
    *mlo = *mhi = 0;
    if (k0 > k1) return false;
    const int lo = band_query_lo(m, k0), hi = band_query_hi(m, k1);
    if (hi <= lo) return false;
    *mlo = lo / bm;
    *mhi = (hi + bm - 1) / bm;
    return true;
}

// ---------------------------------------------------------------------------
// Block masks (dense problems): a byte per (query block, key block) of 128 x
// 128, block_mask[mask_head][qb][kb] != 0 keeps the block (FlashAttention-4
// paper, Section 4: block-sparse patterns are one of the composable
// primitives). The scans below are warp-cooperative: every lane of the calling
// warp must call them with the same arguments, and every lane gets the result.
#ifdef __CUDACC__
// The first block kb' in [kb, hi) with row0[kb'] or row1[kb'] nonzero (row1
// may be null), or hi.
__device__ __forceinline__ int sparse_next(const unsigned char* row0, const unsigned char* row1, int kb, int hi,
                                           int lane) {
    for (int base = kb; base < hi; base += 32) {
        const int c = base + lane;
        const bool a = c < hi && (row0[c] | (row1 ? row1[c] : 0));
        const unsigned m = __ballot_sync(0xffffffffu, a);
        if (m) return base + __ffs(m) - 1;
    }
    return hi;
}

// Number of blocks kb' in [lo, hi) with row0[kb'] or row1[kb'] nonzero.
__device__ __forceinline__ int sparse_count(const unsigned char* row0, const unsigned char* row1, int lo, int hi,
                                            int lane) {
    int n = 0;
    for (int base = lo; base < hi; base += 32) {
        const int c = base + lane;
        const bool a = c < hi && (row0[c] | (row1 ? row1[c] : 0));
        n += __popc(__ballot_sync(0xffffffffu, a));
    }
    return n;
}

// Column scans (the backward's query blocks of one key block): entries
// col[m * stride] for m in [m, hi).
__device__ __forceinline__ int sparse_next_col(const unsigned char* col, long stride, int m, int hi, int lane) {
    for (int base = m; base < hi; base += 32) {
        const int r = base + lane;
        const bool a = r < hi && col[(long)r * stride];
        const unsigned msk = __ballot_sync(0xffffffffu, a);
        if (msk) return base + __ffs(msk) - 1;
    }
    return hi;
}

__device__ __forceinline__ int sparse_count_col(const unsigned char* col, long stride, int lo, int hi, int lane) {
    int n = 0;
    for (int base = lo; base < hi; base += 32) {
        const int r = base + lane;
        n += __popc(__ballot_sync(0xffffffffu, r < hi && col[(long)r * stride]));
    }
    return n;
}
#endif
