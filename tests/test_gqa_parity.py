"""Grouped key/value heads (multi-query and grouped-query attention): the CUDA
path through attn_fwd_gqa / attn_bwd_gqa vs the fp64 oracle.

K and V have Hkv heads; query head h reads key/value head h // (H // Hkv),
and dK, dV of a key/value head sum over the query heads that read it. Small
problems are compared over every element; the workload shape (B2 H16 L8192
with 2 key/value heads, groups of 8) on sampled rows, dK and dV of one
key/value head against the oracle run on its whole group of query heads.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_fwd_close, assert_grad_close, to64

pytestmark = pytest.mark.gpu


def _run(t, causal, scale, deterministic=False, cu=None, grad=True):
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    cud = None if cu is None else cu.cuda()
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale, cu_seqlens=cud)
    if not grad:
        binding.check_status()
        return o, lse
    dq, dk, dv = binding.backward(q, k, v, o, lse, t["do"].cuda(), causal=causal, scale=scale, cu_seqlens=cud,
                                  deterministic=deterministic)
    binding.check_status()
    return o, lse, dq, dk, dv


def _full_check(t, causal, scale, what, deterministic=False, cu=None):
    o, lse, dq, dk, dv = _run(t, causal, scale, deterministic, cu)
    c = None if cu is None else cu.numpy()
    q, k, v, do = (to64(t[n]) for n in ("q", "k", "v", "do"))
    o_ref, lse_ref = oracle.fwd(q, k, v, scale, causal, cu_seqlens=c)
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, what)
    rq, rk, rv = oracle.bwd(q, k, v, do, scale, causal, cu_seqlens=c)
    assert dk.shape == t["k"].shape and dv.shape == t["v"].shape
    assert_grad_close(to64(dq), rq, f"{what} dQ")
    assert_grad_close(to64(dk), rk, f"{what} dK")
    assert_grad_close(to64(dv), rv, f"{what} dV")


@pytest.mark.parametrize("d", [64, 128, 192, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (6, 1), (8, 2)])
@pytest.mark.parametrize("L", [77, 300])
def test_grouped_full(L, H, Hkv, causal, d):
    t = inputs.small(B=2, H=H, L=L, d=d, seed=41, Hkv=Hkv)
    _full_check(t, causal, float(np.float32(1 / np.sqrt(d))), f"H={H} Hkv={Hkv} L={L} causal={causal} d={d}")


@pytest.mark.parametrize("d", [64, 192])
@pytest.mark.parametrize("deterministic", [False, True])
def test_grouped_unsplit(deterministic, d):
    """5 x 8 key blocks x 16 key/value heads = 640 work tiles: one tile per key
    block carries the whole group (the small problems above split the group
    over tiles with partial dK/dV slots; the B2 L8192 workload below splits it
    in part, 4 tiles of 2 heads)."""
    t = inputs.small(B=5, H=32, L=1024, d=d, seed=48, Hkv=16)
    _full_check(t, True, 0.1, f"unsplit det={deterministic} d={d}", deterministic=deterministic)


@pytest.mark.parametrize("d", [128, 192])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_deterministic(causal, d):
    t = inputs.small(B=1, H=8, L=520, d=d, seed=42, Hkv=2)
    _full_check(t, causal, 0.09, f"deterministic causal={causal} d={d}", deterministic=True)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(200, 77), (77, 300), (384, 129)])
def test_grouped_rectangular(Lq, Lk, causal):
    t = inputs.small(B=2, H=6, L=Lq, Lk=Lk, d=128, seed=43, Hkv=3)
    _full_check(t, causal, 0.125, f"Lq={Lq} Lk={Lk} causal={causal}")


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("deterministic", [False, True])
def test_grouped_varlen(deterministic, d):
    lens = [1, 128, 200, 513, 77, 256]
    cu = inputs.cu_seqlens(lens)
    T, H, Hkv = int(cu[-1]), 4, 2
    g = torch.Generator("cpu").manual_seed(44)
    t = {"q": torch.randn(T, H, d, generator=g).to(torch.bfloat16),
         "k": torch.randn(T, Hkv, d, generator=g).to(torch.bfloat16),
         "v": torch.randn(T, Hkv, d, generator=g).to(torch.bfloat16),
         "do": torch.randn(T, H, d, generator=g).to(torch.bfloat16)}
    _full_check(t, True, 0.1, f"varlen d={d} det={deterministic}", deterministic=deterministic, cu=cu)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_value_head_dim_forward(causal):
    """q/k head dim 192, v head dim 128, 6 query heads over 2 key/value heads."""
    t = inputs.small(B=2, H=6, L=300, d=192, dv=128, seed=45, Hkv=2)
    o, lse = _run(t, causal, 0.07, grad=False)
    assert o.shape == (2, 300, 6, 128)
    o_ref, lse_ref = oracle.fwd(*(to64(t[n]) for n in ("q", "k", "v")), 0.07, causal)
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, f"d192/dv128 grouped causal={causal}")


def test_dk_dv_repeatable_without_deterministic_mode():
    """dK and dV take no atomics (one tile accumulates a key block's group, or
    split tiles write slots summed in slot order), so they repeat bit for bit
    even when dQ's accumulation order varies."""
    t = inputs.small(B=2, H=8, L=1024, d=128, seed=46, Hkv=1)
    first = _run(t, True, 0.088)
    for _ in range(3):
        again = _run(t, True, 0.088)
        assert torch.equal(first[3], again[3]) and torch.equal(first[4], again[4])
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])


def test_multi_query_equals_repeated_heads():
    """One key/value head read by every query head gives the result of
    multi-head attention on K, V repeated per head (dK, dV: summed over heads)."""
    t = inputs.small(B=1, H=4, L=333, d=64, seed=47, Hkv=1)
    o, lse, dq, dk, dv = _run(t, True, 0.125)
    rep = {n: t[n].repeat_interleave(4, dim=2) if n in ("k", "v") else t[n] for n in t}
    o2, lse2, dq2, dk2, dv2 = _run(rep, True, 0.125)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert_grad_close(to64(dq), to64(dq2), "MQA vs repeated dQ")
    assert_grad_close(to64(dk), to64(dk2.float().sum(dim=2, keepdim=True)), "MQA vs repeated dK")
    assert_grad_close(to64(dv), to64(dv2.float().sum(dim=2, keepdim=True)), "MQA vs repeated dV")


# ------------------------------------------------------------------ workload shape, sampled rows

GQA8 = inputs.HDSWEEP.with_(name="b2h16kv2l8192d128", hkv=2)


def _rows(L, n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(L, size=n, replace=False).tolist()) | {0, 127, 128, L - 1}
    return sorted(rows)


def test_workload_grouped_b2h16kv2l8192():
    """B2 H16 L8192 d128, 2 key/value heads (groups of 8), causal, spiky K."""
    w = GQA8
    t = inputs.make(w)
    o, lse, dq, dk, dv = _run(t, True, w.scale)
    G = w.H // w.H_kv
    bsel = [0, w.B - 1]
    qrows = _rows(w.L, 16, w.seed)
    # forward and dQ: query heads 3 and 12 (key/value heads 0 and 1), one key/value head per query head
    qh = [3, 12]
    sub = {n: to64(t[n][bsel][:, :, qh]) for n in ("q", "do")}
    sub.update({n: to64(t[n][bsel][:, :, [h // G for h in qh]]) for n in ("k", "v")})
    o_ref, lse_ref = oracle.fwd(sub["q"], sub["k"], sub["v"], w.scale, True, rows=qrows)
    assert_fwd_close(to64(o[bsel][:, qrows][:, :, qh]), to64(lse[bsel][:, qh][:, :, qrows]),
                     o_ref[:, qrows], lse_ref[:, :, qrows], "grouped workload forward")
    rq, _, _ = oracle.bwd(sub["q"], sub["k"], sub["v"], sub["do"], w.scale, True, qrows=qrows, krows=[])
    assert_grad_close(to64(dq[bsel][:, qrows][:, :, qh]), rq[:, qrows], "grouped workload dQ")
    # dK, dV of key/value head 1: the oracle on its whole group of query heads
    kh = 1
    grp = list(range(kh * G, kh * G + G))
    krows = _rows(w.L, 8, w.seed + 1)
    full = {n: to64(t[n][bsel][:, :, grp]) for n in ("q", "do")}
    full.update({n: to64(t[n][bsel][:, :, [kh]]) for n in ("k", "v")})
    _, rk, rv = oracle.bwd(full["q"], full["k"], full["v"], full["do"], w.scale, True, qrows=[], krows=krows)
    assert_grad_close(to64(dk[bsel][:, krows][:, :, [kh]]), rk[:, krows], "grouped workload dK")
    assert_grad_close(to64(dv[bsel][:, krows][:, :, [kh]]), rv[:, krows], "grouped workload dV")
