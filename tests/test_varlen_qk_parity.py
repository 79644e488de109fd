"""Packed sequences with key lengths of their own (attn_fwd_varlen /
attn_bwd_varlen) vs the fp64 oracle.

Sequence b has Lq_b queries (offsets cu_seqlens_q) and Lk_b keys (offsets
cu_seqlens_k) and is its own rectangular problem, causal bottom-right aligned
within it. Cases: longer, shorter, equal and empty sides, ragged tails, every
head dim, grouped heads, the deterministic mode, and a prefill/decode mix.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_fwd_close, assert_grad_close, to64

pytestmark = pytest.mark.gpu

LQ = [1, 128, 200, 513, 77, 256, 0, 300]
LK = [300, 1, 200, 129, 513, 0, 77, 256]


def _problem(lq, lk, H, Hkv, d, seed):
    cu, cuk = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    g = torch.Generator("cpu").manual_seed(seed)
    Tq, Tk = int(cu[-1]), int(cuk[-1])
    t = {"q": torch.randn(Tq, H, d, generator=g).to(torch.bfloat16),
         "k": torch.randn(Tk, Hkv, d, generator=g).to(torch.bfloat16),
         "v": torch.randn(Tk, Hkv, d, generator=g).to(torch.bfloat16),
         "do": torch.randn(Tq, H, d, generator=g).to(torch.bfloat16)}
    return t, cu, cuk


def _run(t, cu, cuk, causal, scale, deterministic=False, grad=True):
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    cq, ck = cu.cuda(), cuk.cuda()
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale, cu_seqlens=cq, cu_seqlens_k=ck)
    if not grad:
        binding.check_status()
        return o, lse
    dq, dk, dv = binding.backward(q, k, v, o, lse, t["do"].cuda(), causal=causal, scale=scale, cu_seqlens=cq,
                                  cu_seqlens_k=ck, deterministic=deterministic)
    binding.check_status()
    return o, lse, dq, dk, dv


def _full_check(t, cu, cuk, causal, scale, what, deterministic=False):
    o, lse, dq, dk, dv = _run(t, cu, cuk, causal, scale, deterministic)
    q, k, v, do = (to64(t[n]) for n in ("q", "k", "v", "do"))
    c, ck = cu.numpy(), cuk.numpy()
    o_ref, lse_ref = oracle.fwd(q, k, v, scale, causal, cu_seqlens=c, cu_seqlens_k=ck)
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, what)
    rq, rk, rv = oracle.bwd(q, k, v, do, scale, causal, cu_seqlens=c, cu_seqlens_k=ck)
    assert_grad_close(to64(dq), rq, f"{what} dQ")
    assert_grad_close(to64(dk), rk, f"{what} dK")
    assert_grad_close(to64(dv), rv, f"{what} dV")


@pytest.mark.parametrize("d", [64, 128, 192, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_separate_lengths_full(causal, d):
    t, cu, cuk = _problem(LQ, LK, 2, 2, d, 61)
    _full_check(t, cu, cuk, causal, float(np.float32(1 / np.sqrt(d))), f"causal={causal} d={d}")


@pytest.mark.parametrize("d", [128, 192])
@pytest.mark.parametrize("deterministic", [False, True])
def test_separate_lengths_grouped(deterministic, d):
    t, cu, cuk = _problem(LK, LQ, 4, 2, d, 62)   # the lengths swapped
    _full_check(t, cu, cuk, True, 0.09, f"grouped det={deterministic} d={d}", deterministic=deterministic)


def test_same_offsets_match_the_shared_array_call():
    """cu_seqlens_k equal to cu_seqlens gives bit for bit the one-array call."""
    lens = [77, 300, 1, 513]
    t, cu, _ = _problem(lens, lens, 2, 2, 128, 63)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    cq = cu.cuda()
    o1, l1 = binding.forward(q, k, v, causal=True, scale=0.1, cu_seqlens=cq)
    o2, l2 = binding.forward(q, k, v, causal=True, scale=0.1, cu_seqlens=cq, cu_seqlens_k=cu.clone().cuda())
    binding.check_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_prefill_decode_mix():
    """Decode steps (1-16 new queries against a long cache) packed with
    prefill sequences (queries = keys), causal, grouped heads."""
    lq = [1, 2048, 16, 1, 777, 4, 1]
    lk = [4096, 2048, 3000, 129, 777, 8192, 1]
    t, cu, cuk = _problem(lq, lk, 8, 2, 128, 64)
    _full_check(t, cu, cuk, True, 0.088, "prefill/decode mix")


def test_argument_errors():
    t, cu, cuk = _problem([3, 4], [5, 6], 2, 2, 64, 65)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(2, q.shape[0], dtype=torch.float32, device="cuda")
    rc = binding.attn_fwd_varlen(q, k, v, o, lse, 2, 2, 2, q.shape[0], k.shape[0], 64, 64, 0.1, True, cu.cuda(),
                                 None)
    assert rc == binding.ATTN_ERR_ARG


def test_workload_prefill_decode_mix():
    """The benchmark's mix: 16 prefill sequences (256-8192 rows) and 16 decode
    steps (1-16 queries against 1024-16384 keys), H16 over 4 key/value heads,
    d128, causal; sampled query and key rows of four sequences against the
    oracle, dK/dV on the whole group of key/value head 1."""
    w = inputs.PREFILL_DECODE
    t = inputs.make(w)
    cu, cuk = t["cu_seqlens"], t["cu_seqlens_k"]
    o, lse, dq, dk, dv = _run(t, cu, cuk, True, w.scale)
    lq, lk = np.diff(cu.numpy()), np.diff(cuk.numpy())
    G = w.H // w.H_kv
    prefill = [b for b in range(w.B) if lq[b] == lk[b]]
    decode = [b for b in range(w.B) if lq[b] != lk[b]]
    picks = [max(prefill, key=lambda b: lq[b]), min(prefill, key=lambda b: lq[b]),
             max(decode, key=lambda b: lk[b]), max(decode, key=lambda b: lq[b])]
    rng = np.random.default_rng(7)
    for b in picks:
        a, c, L, M = int(cu[b]), int(cuk[b]), int(lq[b]), int(lk[b])
        qrows = sorted(set(rng.choice(L, size=min(L, 12), replace=False).tolist()) | {0, L - 1})
        krows = sorted(set(rng.choice(M, size=min(M, 8), replace=False).tolist()) | {0, M - 1})
        kh = 1
        grp = list(range(kh * G, kh * G + G))
        sub = {n: to64(t[n][a:a + L][:, grp])[None] for n in ("q", "do")}
        sub.update({n: to64(t[n][c:c + M][:, [kh]])[None] for n in ("k", "v")})
        o_ref, lse_ref = oracle.fwd(sub["q"], sub["k"], sub["v"], w.scale, True, rows=qrows)
        assert_fwd_close(to64(o[a:a + L][qrows][:, grp])[None], to64(lse[grp][:, a:a + L][:, qrows])[None],
                         o_ref[:, qrows], lse_ref[:, :, qrows], f"mix seq {b} (Lq={L}, Lk={M})")
        rq, rk, rv = oracle.bwd(sub["q"], sub["k"], sub["v"], sub["do"], w.scale, True, qrows=qrows, krows=krows)
        assert_grad_close(to64(dq[a:a + L][qrows][:, grp])[None], rq[:, qrows], f"mix seq {b} dQ")
        assert_grad_close(to64(dk[c:c + M][krows][:, [kh]])[None], rk[:, krows], f"mix seq {b} dK")
        assert_grad_close(to64(dv[c:c + M][krows][:, [kh]])[None], rv[:, krows], f"mix seq {b} dV")
