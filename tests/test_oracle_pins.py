"""Pins for the fp64 oracle, independent of the oracle itself.

Each check ties the oracle to something other than its own formulas: a
hand-derived example (tests/golden/hand_2x2.txt), closed forms of special
cases, a textbook softmax written with scipy on tiny inputs, invariants of
softmax attention, and central finite differences for the backward pass.
The mutant test (test_oracle_mutants.py) shows that plausible mistakes in the
oracle source fail at least one of these.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
from exact_attention_blackwell_tma_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- golden file

def load_golden(name):
    consts = {"LN2": math.log(2.0), "LN3": math.log(3.0)}
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            nums = []
            for tok in val.split(","):
                tok = tok.strip()
                if not tok:
                    continue
                factor = 1.0
                if "*" in tok:
                    a, b = tok.split("*")
                    tok, factor = a.strip(), consts[b.strip()]
                nums.append((consts[tok] if tok in consts else float(tok)) * factor)
            out[key] = np.array(nums)
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_golden_hand_example(causal):
    g = load_golden("hand_2x2.txt")
    shp = (1, 2, 1, 2)
    q, k, v, do = (g[n].reshape(shp) for n in ("q", "k", "v", "do"))
    scale = float(g["scale"][0])
    tag = "causal" if causal else "noncausal"
    o, lse = oracle.fwd(q, k, v, scale, causal)
    np.testing.assert_allclose(o.reshape(-1), g[f"{tag}.o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(-1), g[f"{tag}.lse"], rtol=0, atol=1e-12)
    dq, dk, dv = oracle.bwd(q, k, v, do, scale, causal)
    np.testing.assert_allclose(dq.reshape(-1), g[f"{tag}.dq"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.reshape(-1), g[f"{tag}.dk"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.reshape(-1), g[f"{tag}.dv"], rtol=0, atol=1e-12)


# ------------------------------------------------------------- forward pins

def textbook(q, k, v, scale, causal):
    """softmax(scale Q K^T [+ bottom-right causal mask]) V with scipy, tiny sizes."""
    B, Lq, H, d = q.shape
    Lk = k.shape[1]
    s = np.einsum("bihc,bjhc->bhij", q, k) * scale
    if causal:
        i = np.arange(Lq)[:, None]
        j = np.arange(Lk)[None, :]
        s = np.where(j <= i + (Lk - Lq), s, -np.inf)
    with np.errstate(invalid="ignore"):
        lse = logsumexp(s, axis=-1)
        p = softmax(s, axis=-1)
    p = np.nan_to_num(p, nan=0.0)
    o = np.einsum("bhij,bjhc->bihc", p, v)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Lq,Lk,d", [(1, 1, 1, 1, 1), (2, 3, 5, 5, 4), (1, 2, 7, 11, 8),
                                         (2, 1, 9, 4, 3), (1, 2, 16, 16, 16)])
def test_fwd_matches_textbook_softmax(B, H, Lq, Lk, d, causal):
    q, k, v = rnd((B, Lq, H, d), 1), rnd((B, Lk, H, d), 2), rnd((B, Lk, H, d), 3)
    scale = 0.7
    o, lse = oracle.fwd(q, k, v, scale, causal)
    o_ref, lse_ref = textbook(q, k, v, scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Lq,Lk,d,dv", [(2, 3, 5, 5, 4, 3), (1, 2, 7, 11, 6, 9), (1, 1, 9, 4, 5, 2)])
def test_fwd_matches_textbook_softmax_value_dim(B, H, Lq, Lk, d, dv, causal):
    """v (and O) with a head dim of their own, as the FlashAttention-4 paper's
    Section 5.1 measures at d = 192 for q/k and 128 for v."""
    q, k, v = rnd((B, Lq, H, d), 7), rnd((B, Lk, H, d), 8), rnd((B, Lk, H, dv), 9)
    o, lse = oracle.fwd(q, k, v, 0.45, causal)
    o_ref, lse_ref = textbook(q, k, v, 0.45, causal)
    assert o.shape == (B, Lq, H, dv)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=1e-12, atol=1e-12)


def test_single_key_returns_v_row_of_its_own_width():
    q, k, v = rnd((1, 4, 2, 6), 10), rnd((1, 1, 2, 6), 11), rnd((1, 1, 2, 3), 12)
    o, _ = oracle.fwd(q, k, v, 0.5, False)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Hkv,Lq,Lk,d", [(2, 4, 2, 5, 5, 4), (1, 6, 3, 7, 9, 3), (1, 4, 1, 6, 6, 5)])
def test_fwd_grouped_heads_match_textbook(B, H, Hkv, Lq, Lk, d, causal):
    """Grouped key/value heads: query head h reads key/value head h // (H / Hkv).
    The textbook softmax on K and V with each key/value head repeated for the
    query heads of its group gives the same result (Hkv = 1 is multi-query)."""
    q, k, v = rnd((B, Lq, H, d), 13), rnd((B, Lk, Hkv, d), 14), rnd((B, Lk, Hkv, d), 15)
    o, lse = oracle.fwd(q, k, v, 0.55, causal)
    g = H // Hkv
    o_ref, lse_ref = textbook(q, np.repeat(k, g, axis=2), np.repeat(v, g, axis=2), 0.55, causal)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=1e-12, atol=1e-12)


def test_single_key_returns_v():
    q, k, v = rnd((2, 6, 3, 8), 4), rnd((2, 1, 3, 8), 5), rnd((2, 1, 3, 8), 6)
    s = 0.3 * np.einsum("bihc,bhc->bhi", q, k[:, 0])
    o, lse = oracle.fwd(q, k, v, 0.3, False)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, s, rtol=1e-13, atol=1e-13)   # LSE of one score is it
    # causal, bottom-right aligned: only the last query row sees the single key
    o, lse = oracle.fwd(q, k, v, 0.3, True)
    np.testing.assert_allclose(o[:, -1], v[:, 0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[:, :, -1], s[:, :, -1], rtol=1e-13, atol=1e-13)
    assert np.all(o[:, :-1] == 0) and np.all(np.isneginf(lse[:, :, :-1]))


def test_identical_keys_give_mean_of_v():
    L, d = 9, 5
    q = rnd((1, L, 2, d), 7)
    k = np.broadcast_to(rnd((1, 1, 2, d), 8), (1, L, 2, d)).copy()
    v = rnd((1, L, 2, d), 9)
    o, lse = oracle.fwd(q, k, v, 0.5, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape),
                               rtol=1e-12, atol=1e-12)
    s = 0.5 * np.einsum("bihc,bhc->bhi", q, k[:, 0])
    np.testing.assert_allclose(lse, s + math.log(L), rtol=1e-12, atol=1e-12)


def test_zero_query_gives_column_mean():
    q = np.zeros((1, 4, 1, 6))
    k, v = rnd((1, 10, 1, 6), 10), rnd((1, 10, 1, 6), 11)
    o, lse = oracle.fwd(q, k, v, 1.0, False)
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(v[0, :, 0].mean(0), (4, 6)), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(10), atol=1e-13)


def test_identity_values_expose_probabilities():
    """With V = I (d = Lk), O_i is the probability row P_i: rows sum to 1."""
    L = 12
    q, k = rnd((1, L, 1, L), 12), rnd((1, L, 1, L), 13)
    v = np.eye(L).reshape(1, L, 1, L)
    for causal in (False, True):
        o, _ = oracle.fwd(q, k, v, 0.4, causal)
        p = o[0, :, 0, :]
        np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
        assert (p >= 0).all()
        if causal:
            assert np.all(np.triu(p, 1) == 0)


def test_causal_first_row_returns_v0():
    q, k, v = rnd((2, 8, 3, 4), 14), rnd((2, 8, 3, 4), 15), rnd((2, 8, 3, 4), 16)
    o, lse = oracle.fwd(q, k, v, 0.9, True)
    np.testing.assert_allclose(o[:, 0], v[:, 0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[:, :, 0], 0.9 * np.einsum("bhc,bhc->bh", q[:, 0], k[:, 0]),
                               atol=1e-13)


def test_key_permutation_invariance():
    q, k, v = rnd((1, 6, 2, 4), 17), rnd((1, 10, 2, 4), 18), rnd((1, 10, 2, 4), 19)
    perm = np.random.default_rng(0).permutation(10)
    o1, l1 = oracle.fwd(q, k, v, 0.6, False)
    o2, l2 = oracle.fwd(q, k[:, perm], v[:, perm], 0.6, False)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_causal_row_equals_prefix_attention():
    L = 9
    q, k, v = rnd((1, L, 2, 4), 20), rnd((1, L, 2, 4), 21), rnd((1, L, 2, 4), 22)
    o, lse = oracle.fwd(q, k, v, 0.8, True)
    for i in range(L):
        oi, li = oracle.fwd(q[:, i:i + 1], k[:, :i + 1], v[:, :i + 1], 0.8, False)
        np.testing.assert_allclose(o[:, i], oi[:, 0], atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], li[:, :, 0], atol=1e-13)


def test_bottom_right_causal_with_more_queries():
    """Lq > Lk: rows i < Lq - Lk see no key (O = 0, LSE = -inf)."""
    q, k, v = rnd((1, 7, 1, 3), 23), rnd((1, 4, 1, 3), 24), rnd((1, 4, 1, 3), 25)
    o, lse = oracle.fwd(q, k, v, 1.0, True)
    assert np.all(o[0, :3] == 0) and np.all(np.isneginf(lse[0, 0, :3]))
    assert np.all(np.isfinite(lse[0, 0, 3:]))
    # the last Lk rows behave like square causal attention with the last queries
    o2, l2 = oracle.fwd(q[:, 3:], k, v, 1.0, True)
    np.testing.assert_allclose(o[:, 3:], o2, atol=1e-13)


def test_shift_invariance_of_keys():
    """Adding a vector u to every key shifts row i's scores by scale<q_i,u>:
    probabilities (so O) are unchanged and LSE moves by exactly that amount."""
    q, k, v = rnd((1, 5, 1, 4), 26), rnd((1, 8, 1, 4), 27), rnd((1, 8, 1, 4), 28)
    u = 3.0 * rnd((4,), 29)
    o1, l1 = oracle.fwd(q, k, v, 0.5, False)
    o2, l2 = oracle.fwd(q, k + u, v, 0.5, False)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 0.5 * np.einsum("bihc,c->bhi", q, u), atol=1e-12)


def test_large_scores_do_not_overflow():
    q, k, v = rnd((1, 4, 1, 8), 30), rnd((1, 6, 1, 8), 31), rnd((1, 6, 1, 8), 32)
    o, lse = oracle.fwd(q, k, v, 300.0, False)
    o_ref, lse_ref = textbook(q, k, v, 300.0, False)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12)


def test_varlen_is_per_sequence_attention():
    lens = [3, 1, 6, 4]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, H, d = cu[-1], 2, 4
    q, k, v = rnd((T, H, d), 33), rnd((T, H, d), 34), rnd((T, H, d), 35)
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, 0.7, causal, cu_seqlens=cu)
        for b, L in enumerate(lens):
            a = cu[b]
            ob, lb = textbook(q[None, a:a + L], k[None, a:a + L], v[None, a:a + L], 0.7, causal)
            np.testing.assert_allclose(o[a:a + L], ob[0], atol=1e-12)
            np.testing.assert_allclose(lse[:, a:a + L], lb[0], atol=1e-12)


LENS_Q, LENS_K = [3, 1, 6, 0, 4, 2], [5, 2, 2, 3, 4, 0]   # longer, shorter, equal and empty sides


def _offsets(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def test_varlen_separate_key_lengths_is_per_sequence_attention():
    """With key offsets of their own, sequence b is the rectangular problem of
    its Lq_b queries and Lk_b keys (causal bottom-right aligned within it)."""
    cu, cuk = _offsets(LENS_Q), _offsets(LENS_K)
    H, Hkv, d = 4, 2, 3
    q, k, v = rnd((cu[-1], H, d), 90), rnd((cuk[-1], Hkv, d), 91), rnd((cuk[-1], Hkv, d), 92)
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, 0.6, causal, cu_seqlens=cu, cu_seqlens_k=cuk)
        for b in range(len(LENS_Q)):
            a, L, c, M = cu[b], LENS_Q[b], cuk[b], LENS_K[b]
            if L == 0 or M == 0:
                assert (o[a:a + L] == 0).all() and np.isneginf(lse[:, a:a + L]).all()
                continue
            ob, lb = textbook(q[None, a:a + L], np.repeat(k[None, c:c + M], 2, axis=2),
                              np.repeat(v[None, c:c + M], 2, axis=2), 0.6, causal)
            np.testing.assert_allclose(o[a:a + L], ob[0], atol=1e-12)
            ref = lb[0]
            fin = np.isfinite(ref)
            if fin.any():
                np.testing.assert_allclose(lse[:, a:a + L][fin], ref[fin], atol=1e-12)
            assert np.isneginf(lse[:, a:a + L][~fin]).all()


def textbook_window(q, k, v, scale, wl, wr):
    """softmax over the band i + delta - wl <= j <= i + delta + wr (delta = Lk - Lq,
    -1: no bound), written with scipy on a dense mask, tiny sizes."""
    B, Lq, H, d = q.shape
    Lk = k.shape[1]
    s = np.einsum("bihc,bjhc->bhij", q, k) * scale
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    keep = np.ones((Lq, Lk), dtype=bool)
    if wr >= 0:
        keep &= j <= i + (Lk - Lq) + wr
    if wl >= 0:
        keep &= j >= i + (Lk - Lq) - wl
    s = np.where(keep, s, -np.inf)
    with np.errstate(invalid="ignore"):
        lse = logsumexp(s, axis=-1)
        p = softmax(s, axis=-1)
    p = np.nan_to_num(p, nan=0.0)
    return np.einsum("bhij,bjhc->bihc", p, v), lse


@pytest.mark.parametrize("wl,wr", [(0, 0), (2, 0), (3, 1), (-1, 2), (4, -1), (1, 5)])
@pytest.mark.parametrize("Lq,Lk", [(7, 7), (5, 9), (9, 4)])
def test_window_matches_textbook_band(Lq, Lk, wl, wr):
    """A local window is softmax over a band around the bottom-right diagonal;
    rows whose band holds no key get O = 0 and LSE = -inf."""
    q, k, v = rnd((2, Lq, 2, 3), 80), rnd((2, Lk, 2, 3), 81), rnd((2, Lk, 2, 3), 82)
    o, lse = oracle.fwd(q, k, v, 0.7, False, window_left=wl, window_right=wr)
    o_ref, lse_ref = textbook_window(q, k, v, 0.7, wl, wr)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], atol=1e-12)
    assert np.isneginf(lse[~fin]).all()
    # causal sets the right bound to 0 whatever window_right says
    o_c, _ = oracle.fwd(q, k, v, 0.7, True, window_left=wl, window_right=wr)
    o_c_ref, _ = textbook_window(q, k, v, 0.7, wl, 0)
    np.testing.assert_allclose(o_c, o_c_ref, atol=1e-12)


def test_zero_window_returns_the_diagonal_value():
    """window_left = window_right = 0: row i sees only key i + Lk - Lq, so
    O_i = v_{i + Lk - Lq} and LSE_i = its score; rows with no such key get 0."""
    Lq, Lk = 6, 4
    q, k, v = rnd((1, Lq, 1, 5), 83), rnd((1, Lk, 1, 5), 84), rnd((1, Lk, 1, 5), 85)
    o, lse = oracle.fwd(q, k, v, 0.9, False, window_left=0, window_right=0)
    for i in range(Lq):
        j = i + Lk - Lq
        if 0 <= j < Lk:
            np.testing.assert_allclose(o[0, i, 0], v[0, j, 0], atol=1e-14)
            np.testing.assert_allclose(lse[0, 0, i], 0.9 * q[0, i, 0] @ k[0, j, 0], atol=1e-13)
        else:
            assert (o[0, i, 0] == 0).all() and np.isneginf(lse[0, 0, i])


def test_window_wider_than_the_sequence_is_no_window():
    q, k, v = rnd((1, 8, 2, 4), 86), rnd((1, 8, 2, 4), 87), rnd((1, 8, 2, 4), 88)
    for causal in (False, True):
        a = oracle.fwd(q, k, v, 0.5, causal)
        b = oracle.fwd(q, k, v, 0.5, causal, window_left=8, window_right=8)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


def expand_block_mask(bmask, Lq, Lk, bq, bk):
    """[Hm, nqb, nkb] block mask -> [Hm, Lq, Lk] element mask (numpy repeat)."""
    m = np.repeat(np.repeat(np.asarray(bmask, dtype=bool), bq, axis=1), bk, axis=2)
    return m[:, :Lq, :Lk]


def textbook_masked(q, k, v, scale, keep):
    """softmax over the kept (query, key) pairs; keep is [Hm, Lq, Lk] (Hm 1 or H)."""
    s = np.einsum("bihc,bjhc->bhij", q, k) * scale
    s = np.where(keep[None], s, -np.inf)
    with np.errstate(invalid="ignore"):
        lse = logsumexp(s, axis=-1)
        p = np.nan_to_num(softmax(s, axis=-1), nan=0.0)
    return np.einsum("bhij,bjhc->bihc", p, v), lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bq,bk", [(2, 3), (3, 2), (4, 4)])
@pytest.mark.parametrize("per_head", [False, True])
def test_block_mask_matches_textbook(per_head, bq, bk, causal):
    """A block mask drops whole (query block, key block) rectangles, on top of
    the causal mask; with one mask per head each head uses its own."""
    Lq, Lk, H = 9, 11, 3
    q, k, v = rnd((2, Lq, H, 4), 101), rnd((2, Lk, H, 4), 102), rnd((2, Lk, H, 4), 103)
    nqb, nkb = -(-Lq // bq), -(-Lk // bk)
    bm = (np.random.default_rng(104).random((H if per_head else 1, nqb, nkb)) < 0.6).astype(np.uint8)
    bm[0, 0, :] = 0   # a query block that sees nothing
    o, lse = oracle.fwd(q, k, v, 0.6, causal, block_mask=bm, block=(bq, bk))
    keep = expand_block_mask(bm, Lq, Lk, bq, bk)
    if causal:
        keep = keep & (np.arange(Lk)[None, :] <= np.arange(Lq)[:, None] + (Lk - Lq))[None]
    o_ref, lse_ref = textbook_masked(q, k, v, 0.6, keep)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], atol=1e-12)
    assert np.isneginf(lse[~fin]).all() and (o[:, :bq][:, :, 0] == 0).all()


def test_all_ones_block_mask_is_no_mask():
    q, k, v = rnd((1, 7, 2, 3), 105), rnd((1, 7, 2, 3), 106), rnd((1, 7, 2, 3), 107)
    for causal in (False, True):
        a = oracle.fwd(q, k, v, 0.5, causal)
        b = oracle.fwd(q, k, v, 0.5, causal, block_mask=np.ones((1, 4, 3), np.uint8), block=(2, 3))
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


def test_block_mask_keeping_one_key_block_is_attention_over_it():
    """Every query block keeping only key block c is attention over those keys."""
    Lq, Lk, bq, bk = 8, 9, 4, 3
    q, k, v = rnd((1, Lq, 1, 3), 108), rnd((1, Lk, 1, 3), 109), rnd((1, Lk, 1, 3), 110)
    for c in range(3):
        bm = np.zeros((1, 2, 3), np.uint8)
        bm[0, :, c] = 1
        o, lse = oracle.fwd(q, k, v, 0.7, False, block_mask=bm, block=(bq, bk))
        o_ref, lse_ref = oracle.fwd(q, k[:, c * bk:(c + 1) * bk], v[:, c * bk:(c + 1) * bk], 0.7, False)
        np.testing.assert_allclose(o, o_ref, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-13)


def test_row_subset_matches_full():
    q, k, v = rnd((2, 10, 2, 4), 36), rnd((2, 10, 2, 4), 37), rnd((2, 10, 2, 4), 38)
    full_o, full_l = oracle.fwd(q, k, v, 0.5, True)
    rows = [0, 3, 9]
    o, lse = oracle.fwd(q, k, v, 0.5, True, rows=rows)
    np.testing.assert_array_equal(o[:, rows], full_o[:, rows])
    np.testing.assert_array_equal(lse[:, :, rows], full_l[:, :, rows])
    assert np.isnan(o[:, 1]).all()


def test_workload_inputs_roundtrip_through_oracle():
    """The seeded bf16 inputs widen exactly and the tiny workload runs."""
    t = inputs.make(inputs.TINY)
    q = t["q"].float().numpy()
    assert np.array_equal(q.astype(np.float64).astype(np.float32), q)
    o, lse = oracle.fwd(q, t["k"].float().numpy(), t["v"].float().numpy(),
                        inputs.TINY.scale, False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


# ------------------------------------------------------------- backward pins

def loss(q, k, v, do, scale, causal, cu=None):
    o, _ = oracle.fwd(q, k, v, scale, causal, cu_seqlens=cu)
    return float(np.sum(o * do))


def finite_diff(q, k, v, do, scale, causal, cu=None, h=1e-6):
    grads = []
    for which in range(3):
        arrs = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(arrs[which])
        it = np.nditer(g, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in arrs]
            minus = [a.copy() for a in arrs]
            plus[which][idx] += h
            minus[which][idx] -= h
            g[idx] = (loss(*plus, do, scale, causal, cu) - loss(*minus, do, scale, causal, cu)) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L,d", [(1, 4), (3, 4), (7, 8)])
def test_bwd_finite_differences(L, d, causal):
    q, k, v, do = rnd((1, L, 1, d), 40), rnd((1, L, 1, d), 41), rnd((1, L, 1, d), 42), rnd((1, L, 1, d), 43)
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.6, causal)
    fq, fk, fv = finite_diff(q, k, v, do, 0.6, causal)
    for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
        err = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
        assert err < 1e-6 or np.abs(got - ref).max() < 1e-8, err


def test_bwd_finite_differences_rectangular_and_varlen():
    q, k, v, do = rnd((1, 5, 2, 3), 44), rnd((1, 3, 2, 3), 45), rnd((1, 3, 2, 3), 46), rnd((1, 5, 2, 3), 47)
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.9, True)
    fq, fk, fv = finite_diff(q, k, v, do, 0.9, True)
    for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
        assert np.abs(got - ref).max() < 1e-7
    lens = [2, 3]
    cu = np.array([0, 2, 5], dtype=np.int32)
    q, k, v, do = rnd((5, 1, 3), 48), rnd((5, 1, 3), 49), rnd((5, 1, 3), 50), rnd((5, 1, 3), 51)
    for causal in (False, True):
        dq, dk, dv = oracle.bwd(q, k, v, do, 0.8, causal, cu_seqlens=cu)
        fq, fk, fv = finite_diff(q, k, v, do, 0.8, causal, cu=cu)
        for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
            assert np.abs(got - ref).max() < 1e-7
    assert sum(lens) == 5


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_finite_differences_varlen_separate_keys(causal):
    """Packed sequences whose key lengths differ from their query lengths."""
    cu, cuk = _offsets([2, 3, 1]), _offsets([3, 1, 2])
    q, do = rnd((cu[-1], 2, 3), 93), rnd((cu[-1], 2, 3), 94)
    k, v = rnd((cuk[-1], 1, 3), 95), rnd((cuk[-1], 1, 3), 96)
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.8, causal, cu_seqlens=cu, cu_seqlens_k=cuk)
    assert dk.shape == k.shape

    def loss2(q_, k_, v_):
        o, _ = oracle.fwd(q_, k_, v_, 0.8, causal, cu_seqlens=cu, cu_seqlens_k=cuk)
        return float(np.sum(o * do))

    for got, which in ((dq, 0), (dk, 1), (dv, 2)):
        arrs = [q, k, v]
        g = np.zeros_like(arrs[which])
        for idx in np.ndindex(g.shape):
            plus = [a.copy() for a in arrs]
            minus = [a.copy() for a in arrs]
            plus[which][idx] += 1e-6
            minus[which][idx] -= 1e-6
            g[idx] = (loss2(*plus) - loss2(*minus)) / 2e-6
        assert np.abs(got - g).max() < 1e-7


@pytest.mark.parametrize("wl,wr", [(1, 0), (2, 1), (0, -1)])
def test_bwd_finite_differences_window(wl, wr):
    q, k, v, do = rnd((1, 6, 2, 3), 97), rnd((1, 5, 2, 3), 98), rnd((1, 5, 2, 3), 99), rnd((1, 6, 2, 3), 100)
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.8, False, window_left=wl, window_right=wr)

    def loss_w(q_, k_, v_):
        o, _ = oracle.fwd(q_, k_, v_, 0.8, False, window_left=wl, window_right=wr)
        return float(np.sum(o * do))

    for got, which in ((dq, 0), (dk, 1), (dv, 2)):
        arrs = [q, k, v]
        g = np.zeros_like(arrs[which])
        for idx in np.ndindex(g.shape):
            plus = [a.copy() for a in arrs]
            minus = [a.copy() for a in arrs]
            plus[which][idx] += 1e-6
            minus[which][idx] -= 1e-6
            g[idx] = (loss_w(*plus) - loss_w(*minus)) / 2e-6
        assert np.abs(got - g).max() < 1e-7


@pytest.mark.parametrize("per_head", [False, True])
def test_bwd_finite_differences_block_mask(per_head):
    H = 2
    q, k, v, do = rnd((1, 6, H, 3), 111), rnd((1, 5, H, 3), 112), rnd((1, 5, H, 3), 113), rnd((1, 6, H, 3), 114)
    bm = np.array([[[1, 0, 1], [0, 1, 1], [1, 1, 0]]], np.uint8)
    if per_head:
        bm = np.concatenate([bm, bm[:, ::-1]], axis=0)
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.8, True, block_mask=bm, block=(2, 2))

    def loss_b(q_, k_, v_):
        o, _ = oracle.fwd(q_, k_, v_, 0.8, True, block_mask=bm, block=(2, 2))
        return float(np.sum(o * do))

    for got, which in ((dq, 0), (dk, 1), (dv, 2)):
        arrs = [q, k, v]
        g = np.zeros_like(arrs[which])
        for idx in np.ndindex(g.shape):
            plus = [a.copy() for a in arrs]
            minus = [a.copy() for a in arrs]
            plus[which][idx] += 1e-6
            minus[which][idx] -= 1e-6
            g[idx] = (loss_b(*plus) - loss_b(*minus)) / 2e-6
        assert np.abs(got - g).max() < 1e-7


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_finite_differences_value_dim(causal):
    q, k = rnd((1, 5, 2, 4), 60), rnd((1, 6, 2, 4), 61)
    v, do = rnd((1, 6, 2, 3), 62), rnd((1, 5, 2, 3), 63)
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.7, causal)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    fq, fk, fv = finite_diff(q, k, v, do, 0.7, causal)
    for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
        assert np.abs(got - ref).max() < 1e-7


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_finite_differences_grouped_heads(causal):
    """dK and dV of a key/value head sum over the query heads of its group."""
    q, k = rnd((1, 5, 4, 3), 64), rnd((1, 6, 2, 3), 65)
    v, do = rnd((1, 6, 2, 3), 66), rnd((1, 5, 4, 3), 67)
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.8, causal)
    assert dk.shape == k.shape and dv.shape == v.shape
    fq, fk, fv = finite_diff(q, k, v, do, 0.8, causal)
    for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
        assert np.abs(got - ref).max() < 1e-7


def test_bwd_column_sums():
    """sum_j dS_ij = 0 gives sum_j dK_j = 0; rows of P sum to 1 give
    sum_j dV_j = sum_i dO_i (per batch and head)."""
    q, k, v, do = (rnd((2, 12, 3, 5), s) for s in (52, 53, 54, 55))
    for causal in (False, True):
        dq, dk, dv = oracle.bwd(q, k, v, do, 0.7, causal)
        np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
        np.testing.assert_allclose(dv.sum(axis=1), do.sum(axis=1), atol=1e-12)


def test_bwd_single_key():
    """One key: P = 1, so dS = 0 => dQ = dK = 0, and dV_0 = sum_i dO_i."""
    q, k, v, do = rnd((1, 6, 2, 4), 56), rnd((1, 1, 2, 4), 57), rnd((1, 1, 2, 4), 58), rnd((1, 6, 2, 4), 59)
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.5, False)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)
    np.testing.assert_allclose(dv[:, 0], do.sum(axis=1), atol=1e-13)


def test_bwd_row_subsets_match_full():
    q, k, v, do = (rnd((1, 16, 2, 4), s) for s in (60, 61, 62, 63))
    for causal in (False, True):
        fq, fk, fv = oracle.bwd(q, k, v, do, 0.5, causal)
        dq, dk, dv = oracle.bwd(q, k, v, do, 0.5, causal, qrows=[2, 15], krows=[0, 7, 14])
        np.testing.assert_array_equal(dq[:, [2, 15]], fq[:, [2, 15]])
        np.testing.assert_array_equal(dk[:, [0, 7, 14]], fk[:, [0, 7, 14]])
        np.testing.assert_array_equal(dv[:, [0, 7, 14]], fv[:, [0, 7, 14]])
        dq, dk, dv = oracle.bwd(q, k, v, do, 0.5, causal, qrows=[], krows=[13])
        np.testing.assert_array_equal(dk[:, 13], fk[:, 13])
        assert np.isnan(dq).all()
