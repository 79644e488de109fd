"""Block masks through attn_fwd_ex / attn_bwd_ex vs the fp64 oracle.

A byte mask [Hm, ceil(Lq/128), ceil(Lk/128)] (Hm 1 or H) drops whole
128 x 128 blocks of (query, key) pairs on top of the causal or window mask.
Cases: random masks with query blocks and key blocks that keep nothing,
shared and per-head masks, every head dim, d_qk 192 / d_v 128, grouped heads,
windows, the deterministic mode (its semaphores count only the kept key
blocks), and a local-plus-strided pattern at the B2 H16 L8192 shape.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_fwd_close, assert_grad_close, to64

pytestmark = pytest.mark.gpu


def random_mask(Hm, Lq, Lk, seed, density=0.5):
    nq, nk = -(-Lq // 128), -(-Lk // 128)
    m = (np.random.default_rng(seed).random((Hm, nq, nk)) < density).astype(np.uint8)
    if nq > 1:
        m[0, 1, :] = 0          # a query block that keeps nothing
    if nk > 2:
        m[:, :, 2] = 0          # a key block nobody keeps
    return m


def _run(t, causal, scale, mask, window=(-1, -1), deterministic=False, grad=True):
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    bm = torch.from_numpy(mask).cuda()
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale, window=window, block_mask=bm)
    if not grad:
        binding.check_status()
        return o, lse
    dq, dk, dv = binding.backward(q, k, v, o, lse, t["do"].cuda(), causal=causal, scale=scale, window=window,
                                  block_mask=bm, deterministic=deterministic)
    binding.check_status()
    return o, lse, dq, dk, dv


def _full_check(t, causal, scale, mask, what, window=(-1, -1), deterministic=False):
    o, lse, dq, dk, dv = _run(t, causal, scale, mask, window, deterministic)
    q, k, v, do = (to64(t[n]) for n in ("q", "k", "v", "do"))
    kw = dict(window_left=window[0], window_right=window[1], block_mask=mask)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale, causal, **kw)
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, what)
    rq, rk, rv = oracle.bwd(q, k, v, do, scale, causal, **kw)
    assert_grad_close(to64(dq), rq, f"{what} dQ")
    assert_grad_close(to64(dk), rk, f"{what} dK")
    assert_grad_close(to64(dv), rv, f"{what} dV")


@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 192, 256])
def test_block_mask_full(d, causal, per_head):
    t = inputs.small(B=2, H=2, L=700, d=d, seed=81)
    mask = random_mask(2 if per_head else 1, 700, 700, 82 + d)
    _full_check(t, causal, float(np.float32(1 / np.sqrt(d))), mask, f"d={d} causal={causal} per_head={per_head}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Lq,Lk", [(300, 900), (900, 300), (129, 1)])
def test_block_mask_rectangular(Lq, Lk, d):
    """Odd query-block counts leave the last 256-row tile one 128-row block."""
    t = inputs.small(B=1, H=2, L=Lq, Lk=Lk, d=d, seed=83)
    _full_check(t, True, 0.1, random_mask(2, Lq, Lk, 84, 0.7), f"Lq={Lq} Lk={Lk} d={d}")


@pytest.mark.parametrize("d", [64, 128])
def test_block_mask_with_window(d):
    t = inputs.small(B=1, H=2, L=1000, d=d, seed=85)
    _full_check(t, True, 0.09, random_mask(1, 1000, 1000, 86, 0.6), f"mask + window d={d}", window=(300, 0))


@pytest.mark.parametrize("deterministic", [False, True])
def test_block_mask_grouped_heads(deterministic):
    t = inputs.small(B=1, H=8, L=900, d=128, seed=87, Hkv=2)
    _full_check(t, True, 0.08, random_mask(8, 900, 900, 88, 0.6), f"grouped det={deterministic}",
                deterministic=deterministic)


def test_block_mask_value_head_dim():
    t = inputs.small(B=2, H=2, L=500, d=192, dv=128, seed=89)
    _full_check(t, False, 0.07, random_mask(2, 500, 500, 90), "d192/dv128")


def test_all_ones_block_mask_matches_no_mask():
    t = inputs.small(B=1, H=2, L=600, d=128, seed=91)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = binding.forward(q, k, v, causal=True, scale=0.1)
    ones = torch.ones(1, 5, 5, dtype=torch.uint8, device="cuda")
    o2, l2 = binding.forward(q, k, v, causal=True, scale=0.1, block_mask=ones)
    binding.check_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_deterministic_block_mask_is_bit_identical():
    t = inputs.small(B=1, H=4, L=2000, d=128, seed=92)
    mask = random_mask(4, 2000, 2000, 93, 0.5)
    ref = _run(t, True, 0.088, mask, deterministic=True)
    for _ in range(3):
        again = _run(t, True, 0.088, mask, deterministic=True)
        for a, b in zip(ref, again):
            assert torch.equal(a, b)


def test_workload_local_strided():
    """B2 H16 L8192 d128 causal with the local-plus-strided block pattern;
    sampled rows of heads 3 and 12."""
    w = inputs.HDSWEEP.with_(block_pattern=("local_strided", 4, 8))
    t = inputs.make(w)
    mask = inputs.block_mask(w).numpy()
    o, lse, dq, dk, dv = _run(t, True, w.scale, mask)
    rng = np.random.default_rng(6)
    qrows = sorted(set(rng.choice(w.L, size=16, replace=False).tolist()) | {0, 127, 128, w.L - 1})
    krows = sorted(set(rng.choice(w.L, size=10, replace=False).tolist()) | {0, 1023, w.L - 1})
    heads = [3, 12]
    sub = {n: to64(t[n][:, :, heads]) for n in ("q", "k", "v", "do")}
    o_ref, lse_ref = oracle.fwd(sub["q"], sub["k"], sub["v"], w.scale, True, rows=qrows, block_mask=mask)
    assert_fwd_close(to64(o[:, qrows][:, :, heads]), to64(lse[:, heads][:, :, qrows]), o_ref[:, qrows],
                     lse_ref[:, :, qrows], "local-strided workload")
    rq, rk, rv = oracle.bwd(sub["q"], sub["k"], sub["v"], sub["do"], w.scale, True, qrows=qrows, krows=krows,
                            block_mask=mask)
    assert_grad_close(to64(dq[:, qrows][:, :, heads]), rq[:, qrows], "local-strided dQ")
    assert_grad_close(to64(dk[:, krows][:, :, heads]), rk[:, krows], "local-strided dK")
    assert_grad_close(to64(dv[:, krows][:, :, heads]), rv[:, krows], "local-strided dV")
