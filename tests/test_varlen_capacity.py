"""Packed batches at the sequence map's capacity -- 1024 sequences, the most
one varlen call takes -- against the fp64 oracle over every element: forward
and backward, both modes, every head dim, single CTAs and CTA pairs, one
offset array and two, grouped heads.

The lengths come from a seeded generator: most sequences are short (0-40 rows,
empty ones included) and every 64th is 129-400 rows long, so the batch spans
many 128-row tiles with ragged tails and the longest-first sequence map orders
all 1024 entries.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_fwd_close, assert_grad_close, to64

pytestmark = pytest.mark.gpu

NSEQ = 1024   # sequences per varlen call (the capacity of the sequence map)


def _lengths(seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 41, size=NSEQ)
    lens[::64] = rng.integers(129, 401, size=NSEQ // 64)
    return [int(x) for x in lens]


def _problem(lq, lk, H, Hkv, d, seed):
    cu, cuk = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    g = torch.Generator("cpu").manual_seed(seed)
    Tq, Tk = int(cu[-1]), int(cuk[-1])
    t = {"q": torch.randn(Tq, H, d, generator=g).to(torch.bfloat16),
         "k": torch.randn(Tk, Hkv, d, generator=g).to(torch.bfloat16),
         "v": torch.randn(Tk, Hkv, d, generator=g).to(torch.bfloat16),
         "do": torch.randn(Tq, H, d, generator=g).to(torch.bfloat16)}
    return t, cu, cuk


def _check(t, cu, cuk, causal, scale, deterministic, what):
    """Forward and backward through the C ABI, every element against the oracle.
    cuk is None for one offset array shared by queries and keys."""
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    cq = cu.cuda()
    ck = cuk.cuda() if cuk is not None else None
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale, cu_seqlens=cq, cu_seqlens_k=ck)
    dq, dk, dv = binding.backward(q, k, v, o, lse, do, causal=causal, scale=scale, cu_seqlens=cq,
                                  cu_seqlens_k=ck, deterministic=deterministic)
    binding.check_status()
    q64, k64, v64, do64 = (to64(t[n]) for n in ("q", "k", "v", "do"))
    c = cu.numpy()
    c_k = cuk.numpy() if cuk is not None else None
    o_ref, lse_ref = oracle.fwd(q64, k64, v64, scale, causal, cu_seqlens=c, cu_seqlens_k=c_k)
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, what)
    rq, rk, rv = oracle.bwd(q64, k64, v64, do64, scale, causal, cu_seqlens=c, cu_seqlens_k=c_k)
    assert_grad_close(to64(dq), rq, f"{what} dQ")
    assert_grad_close(to64(dk), rk, f"{what} dK")
    assert_grad_close(to64(dv), rv, f"{what} dV")


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 192, 256])
def test_max_batch(d, causal, deterministic):
    lens = _lengths(71)
    t, cu, _ = _problem(lens, lens, 2, 2, d, 72)
    _check(t, cu, None, causal, float(np.float32(1 / np.sqrt(d))), deterministic,
           f"1024 seqs d={d} causal={causal} det={deterministic}")


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_max_batch_cta_pairs(d, deterministic):
    lens = _lengths(73)
    t, cu, _ = _problem(lens, lens, 4, 2, d, 74)
    prev = binding.attn_set_backward_cta_pairs(1)
    try:
        _check(t, cu, None, True, 0.09, deterministic, f"1024 seqs pairs d={d} det={deterministic}")
    finally:
        binding.attn_set_backward_cta_pairs(prev)


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_max_batch_separate_key_offsets_grouped(causal, deterministic):
    lq, lk = _lengths(75), _lengths(76)
    t, cu, cuk = _problem(lq, lk, 4, 1, 128, 77)
    _check(t, cu, cuk, causal, 0.09, deterministic, f"1024 seqs q/k offsets causal={causal} det={deterministic}")


def test_max_batch_deterministic_is_bit_identical():
    lens = _lengths(78)
    t, cu, _ = _problem(lens, lens, 2, 2, 128, 79)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    cq = cu.cuda()
    o, lse = binding.forward(q, k, v, causal=True, scale=0.09, cu_seqlens=cq)
    ref = binding.backward(q, k, v, o, lse, do, causal=True, scale=0.09, cu_seqlens=cq, deterministic=True)
    for _ in range(2):
        again = binding.backward(q, k, v, o, lse, do, causal=True, scale=0.09, cu_seqlens=cq, deterministic=True)
        for a, b in zip(ref, again):
            assert torch.equal(a, b)
    binding.check_status()
