"""Local (sliding-window) masks through attn_fwd_ex / attn_bwd_ex vs the fp64
oracle.

Query i sees keys i + delta - window_left .. i + delta + window_right (delta =
Lk - Lq, -1: open side; causal sets the right bound to 0). Cases: one- and
two-sided windows narrower and wider than a 128-key block, windows on block
boundaries, the zero window, rectangular problems where rows see nothing,
every head dim, d_qk 192 / d_v 128, grouped heads, varlen with key offsets of
their own, and the deterministic mode (whose per-tile semaphores count only
the key blocks inside the band).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_fwd_close, assert_grad_close, to64

pytestmark = pytest.mark.gpu

WINDOWS = [(0, 0), (5, 0), (127, 0), (128, 0), (200, 0), (64, 64), (-1, 70), (300, -1), (0, -1)]


def _run(t, causal, scale, window, deterministic=False, cu=None, cuk=None, grad=True):
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    cq = None if cu is None else cu.cuda()
    ck = None if cuk is None else cuk.cuda()
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale, cu_seqlens=cq, cu_seqlens_k=ck, window=window)
    if not grad:
        binding.check_status()
        return o, lse
    dq, dk, dv = binding.backward(q, k, v, o, lse, t["do"].cuda(), causal=causal, scale=scale, cu_seqlens=cq,
                                  cu_seqlens_k=ck, deterministic=deterministic, window=window)
    binding.check_status()
    return o, lse, dq, dk, dv


def _full_check(t, causal, scale, window, what, deterministic=False, cu=None, cuk=None):
    o, lse, dq, dk, dv = _run(t, causal, scale, window, deterministic, cu, cuk)
    q, k, v, do = (to64(t[n]) for n in ("q", "k", "v", "do"))
    kw = dict(window_left=window[0], window_right=window[1],
              cu_seqlens=None if cu is None else cu.numpy(), cu_seqlens_k=None if cuk is None else cuk.numpy())
    o_ref, lse_ref = oracle.fwd(q, k, v, scale, causal, **kw)
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, what)
    rq, rk, rv = oracle.bwd(q, k, v, do, scale, causal, **kw)
    assert_grad_close(to64(dq), rq, f"{what} dQ")
    assert_grad_close(to64(dk), rk, f"{what} dK")
    assert_grad_close(to64(dv), rv, f"{what} dV")


@pytest.mark.parametrize("window", WINDOWS, ids=[f"w{a}_{b}" for a, b in WINDOWS])
@pytest.mark.parametrize("d", [64, 128, 192, 256])
def test_window_full(d, window):
    t = inputs.small(B=2, H=2, L=513, d=d, seed=71)
    _full_check(t, False, float(np.float32(1 / np.sqrt(d))), window, f"d={d} window={window}")


@pytest.mark.parametrize("window", [(100, 0), (0, 0), (300, 5)])
@pytest.mark.parametrize("L", [1, 77, 129, 300])
def test_window_ragged_and_causal(L, window):
    """causal with a left window (the causal flag sets the right bound to 0)."""
    t = inputs.small(B=2, H=2, L=L, d=128, seed=72)
    _full_check(t, True, 0.09, window, f"causal L={L} window={window}")


@pytest.mark.parametrize("window", [(50, 0), (0, 30), (200, 200)])
@pytest.mark.parametrize("Lq,Lk", [(300, 77), (77, 300), (513, 129)])
def test_window_rectangular(Lq, Lk, window):
    t = inputs.small(B=1, H=2, L=Lq, Lk=Lk, d=64, seed=73)
    _full_check(t, False, 0.125, window, f"Lq={Lq} Lk={Lk} window={window}")


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("d", [128, 192])
def test_window_grouped_deterministic(d, deterministic):
    t = inputs.small(B=1, H=8, L=1100, d=d, seed=74, Hkv=2)
    _full_check(t, True, 0.08, (300, 0), f"grouped d={d} det={deterministic}", deterministic=deterministic)


def test_window_value_head_dim():
    t = inputs.small(B=2, H=2, L=400, d=192, dv=128, seed=75)
    _full_check(t, False, 0.07, (150, 40), "d192/dv128 window")


@pytest.mark.parametrize("deterministic", [False, True])
def test_window_varlen_separate_keys(deterministic):
    lq, lk = [1, 128, 200, 513, 0, 300, 700], [300, 1, 200, 129, 77, 256, 700]
    cu, cuk = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    g = torch.Generator("cpu").manual_seed(76)
    Tq, Tk = int(cu[-1]), int(cuk[-1])
    t = {"q": torch.randn(Tq, 4, 128, generator=g).to(torch.bfloat16),
         "k": torch.randn(Tk, 2, 128, generator=g).to(torch.bfloat16),
         "v": torch.randn(Tk, 2, 128, generator=g).to(torch.bfloat16),
         "do": torch.randn(Tq, 4, 128, generator=g).to(torch.bfloat16)}
    _full_check(t, True, 0.1, (160, 0), f"varlen window det={deterministic}", deterministic=deterministic,
                cu=cu, cuk=cuk)


def test_deterministic_window_is_bit_identical():
    t = inputs.small(B=1, H=4, L=2048, d=128, seed=77)
    ref = _run(t, True, 0.088, (700, 0), deterministic=True)
    for _ in range(3):
        again = _run(t, True, 0.088, (700, 0), deterministic=True)
        for a, b in zip(ref, again):
            assert torch.equal(a, b)


def test_window_wider_than_the_sequence_matches_no_window():
    t = inputs.small(B=1, H=2, L=600, d=128, seed=78)
    a = _run(t, True, 0.1, (-1, -1), grad=False)
    b = _run(t, True, 0.1, (600, 600), grad=False)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------------------------ workload shape, sampled rows

SLIDING = inputs.HDSWEEP.with_(name="b2h16l8192d128_window4096", window=(4096, 0))


def test_workload_sliding_window():
    """B2 H16 L8192 d128, causal with a 4096-key window, spiky K; sampled rows
    of heads 3 and 12 of both batch entries."""
    w = SLIDING
    t = inputs.make(w)
    o, lse, dq, dk, dv = _run(t, True, w.scale, w.window)
    rng = np.random.default_rng(5)
    qrows = sorted(set(rng.choice(w.L, size=16, replace=False).tolist()) | {0, 4095, 4096, 4097, w.L - 1})
    krows = sorted(set(rng.choice(w.L, size=10, replace=False).tolist()) | {0, 4095, w.L - 1})
    heads = [3, 12]
    sub = {n: to64(t[n][:, :, heads]) for n in ("q", "k", "v", "do")}
    kw = dict(window_left=w.window[0], window_right=w.window[1])
    o_ref, lse_ref = oracle.fwd(sub["q"], sub["k"], sub["v"], w.scale, True, rows=qrows, **kw)
    assert_fwd_close(to64(o[:, qrows][:, :, heads]), to64(lse[:, heads][:, :, qrows]), o_ref[:, qrows],
                     lse_ref[:, :, qrows], "sliding-window workload")
    rq, rk, rv = oracle.bwd(sub["q"], sub["k"], sub["v"], sub["do"], w.scale, True, qrows=qrows, krows=krows, **kw)
    assert_grad_close(to64(dq[:, qrows][:, :, heads]), rq[:, qrows], "sliding-window workload dQ")
    assert_grad_close(to64(dk[:, krows][:, :, heads]), rk[:, krows], "sliding-window workload dK")
    assert_grad_close(to64(dv[:, krows][:, :, heads]), rv[:, krows], "sliding-window workload dV")
