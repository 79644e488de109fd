"""Backward on CTA pairs (2-CTA tensor cores, tcgen05 .cta_group::2) against
the fp64 oracle.

FlashAttention-4 paper, Section 3.2.3: the two CTAs of a cluster run the
backward's MMAs together with M = 256 (each stages half of operand B), and the
pair sums dQ over its 256 keys before one reduce-add pass. The kernel covers
grouped heads (a work tile walks every query head of its
key/value head's group), no mask beyond the causal one and no block mask,
dense or packed, in both modes, head dims 64 and 128 (at 64 the column halves
of operand B are 32 columns with the 64-byte swizzle);
attn_set_backward_cta_pairs switches it on. These tests switch it on and
compare every element with the oracle (ragged lengths that leave the pair's second key block partly or wholly
past the keys, Lq != Lk, packed batches with one or two offset arrays), check
that the deterministic mode repeats bit for bit, that problems the pair kernel
does not cover still come out right with the switch on, and the workload
shapes on sampled rows.
"""
import numpy as np
import pytest
import torch

from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_grad_close, oracle_bwd_subset, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def pairs_on():
    prev = binding.attn_set_backward_cta_pairs(1)
    yield
    binding.attn_set_backward_cta_pairs(prev)


def _grads(t, causal, scale, deterministic=False, cu=None, cuk=None, **kw):
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    cud = cu.cuda() if cu is not None else None
    ckd = cuk.cuda() if cuk is not None else None
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale, cu_seqlens=cud, cu_seqlens_k=ckd, **kw)
    g = binding.backward(q, k, v, o, lse, do, causal=causal, scale=scale, cu_seqlens=cud, cu_seqlens_k=ckd,
                         deterministic=deterministic, **kw)
    binding.check_status()
    return g


def _check(t, causal, scale, what, deterministic=False, cu=None, cuk=None):
    dq, dk, dv = _grads(t, causal, scale, deterministic, cu, cuk)
    import oracle
    rq, rk, rv = oracle.bwd(*(to64(t[n]) for n in ("q", "k", "v", "do")), scale, causal,
                            cu_seqlens=None if cu is None else cu.numpy(),
                            cu_seqlens_k=None if cuk is None else cuk.numpy())
    assert_grad_close(to64(dq), rq, f"{what} dQ")
    assert_grad_close(to64(dk), rk, f"{what} dK")
    assert_grad_close(to64(dv), rv, f"{what} dV")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [1, 77, 128, 129, 256, 300, 513, 1000])
def test_pair_ragged_full(L, causal, deterministic, d):
    t = inputs.small(B=2, H=2, L=L, d=d, seed=41)
    _check(t, causal, 0.088, f"pair d={d} L={L} causal={causal} det={deterministic}", deterministic)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(200, 77), (77, 300), (384, 129), (129, 640), (640, 256)])
def test_pair_rectangular(Lq, Lk, causal, d):
    t = inputs.small(B=1, H=2, L=Lq, Lk=Lk, d=d, seed=42)
    _check(t, causal, 0.088, f"pair d={d} Lq={Lq} Lk={Lk} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_pair_varlen(causal, deterministic, d):
    lens = [1, 128, 200, 513, 77, 256, 384, 0, 129]
    cu = inputs.cu_seqlens(lens)
    g = torch.Generator("cpu").manual_seed(43)
    T = int(cu[-1])
    t = {n: torch.randn(T, 3, d, generator=g).to(torch.bfloat16) for n in ("q", "k", "v", "do")}
    _check(t, causal, 0.09, f"pair d={d} varlen causal={causal} det={deterministic}", deterministic, cu=cu)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_pair_varlen_separate_key_offsets(causal, d):
    lq, lk = [1, 128, 200, 513, 0, 300], [300, 1, 200, 129, 77, 256]
    cu, cuk = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    g = torch.Generator("cpu").manual_seed(44)
    t = {"q": torch.randn(int(cu[-1]), 2, d, generator=g).to(torch.bfloat16),
         "k": torch.randn(int(cuk[-1]), 2, d, generator=g).to(torch.bfloat16),
         "v": torch.randn(int(cuk[-1]), 2, d, generator=g).to(torch.bfloat16),
         "do": torch.randn(int(cu[-1]), 2, d, generator=g).to(torch.bfloat16)}
    _check(t, causal, 0.09, f"pair d={d} varlen q/k offsets causal={causal}", cu=cu, cuk=cuk)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_pair_deterministic_is_bit_identical(causal, d):
    t = inputs.small(B=2, H=4, L=1500, d=d, seed=45)
    ref = _grads(t, causal, 0.088, deterministic=True)
    for _ in range(3):
        again = _grads(t, causal, 0.088, deterministic=True)
        for a, b in zip(ref, again):
            assert torch.equal(a, b)


@pytest.mark.parametrize("d", [64, 128])
def test_pair_agrees_with_single_ctas(d):
    """The same problem on CTA pairs and on single CTAs: dQ sums in another
    order, so the two agree to rounding, both within tolerance of each other."""
    t = inputs.small(B=2, H=3, L=900, d=d, seed=46)
    pair = _grads(t, True, 0.088)
    binding.attn_set_backward_cta_pairs(0)
    single = _grads(t, True, 0.088)
    for name, a, b in zip(("dQ", "dK", "dV"), pair, single):
        assert_grad_close(to64(a), to64(b), f"pair vs single {name}")


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (6, 1), (8, 2)])
@pytest.mark.parametrize("L,d", [(77, 128), (300, 128), (513, 128), (77, 64), (513, 64)])
def test_pair_grouped_heads(L, d, H, Hkv, causal, deterministic):
    """Grouped heads on CTA pairs: a tile's key blocks see every query head of
    the group, and dK/dV sum over them in the tile."""
    t = inputs.small(B=2, H=H, L=L, d=d, seed=48, Hkv=Hkv)
    _check(t, causal, 0.088, f"pair gqa d={d} L={L} H={H}/{Hkv} causal={causal} det={deterministic}", deterministic)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("deterministic", [False, True])
def test_pair_grouped_heads_varlen(deterministic, d):
    lens = [1, 128, 200, 513, 77, 256, 0, 129]
    cu = inputs.cu_seqlens(lens)
    g = torch.Generator("cpu").manual_seed(49)
    T = int(cu[-1])
    t = {"q": torch.randn(T, 6, d, generator=g).to(torch.bfloat16),
         "k": torch.randn(T, 2, d, generator=g).to(torch.bfloat16),
         "v": torch.randn(T, 2, d, generator=g).to(torch.bfloat16),
         "do": torch.randn(T, 6, d, generator=g).to(torch.bfloat16)}
    _check(t, True, 0.09, f"pair gqa d={d} varlen det={deterministic}", deterministic, cu=cu)


@pytest.mark.parametrize("d", [64, 128])
def test_pair_grouped_deterministic_is_bit_identical(d):
    t = inputs.small(B=1, H=8, L=1200, d=d, seed=50, Hkv=2)
    ref = _grads(t, True, 0.088, deterministic=True)
    for _ in range(3):
        again = _grads(t, True, 0.088, deterministic=True)
        for a, b in zip(ref, again):
            assert torch.equal(a, b)


@pytest.mark.parametrize("what", ["window", "blockmask", "d64window", "d192"])
def test_pair_switch_leaves_other_problems_correct(what):
    """With the switch on, problems outside the pair kernel run on single CTAs."""
    import oracle
    d = {"d64window": 64, "d192": 192}.get(what, 128)
    t = inputs.small(B=1, H=2, L=300, d=d, seed=47)
    kw, okw = {}, {}
    if what in ("window", "d64window"):
        kw, okw = {"window": (100, -1)}, {"window_left": 100, "window_right": -1}
    if what == "blockmask":
        m = np.ones((1, 3, 3), np.uint8)
        m[0, 2, 1] = 0
        kw, okw = {"block_mask": torch.from_numpy(m).cuda()}, {"block_mask": m}
    dq, dk, dv = _grads(t, True, 0.1, **kw)
    rq, rk, rv = oracle.bwd(*(to64(t[n]) for n in ("q", "k", "v", "do")), 0.1, True, **okw)
    for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), (rq, rk, rv)):
        assert_grad_close(to64(a), r, f"pair switch {what} {name}")


def _rows(L, n, seed):
    rng = np.random.default_rng(seed)
    return sorted(set(rng.choice(L, size=min(n, L), replace=False).tolist()) | {0, 1, 127, 128, 255, 256, L - 1})


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("wname,causal", [("MHA4K", True), ("MHA4K", False), ("LONG", True), ("LONG", False)])
def test_pair_workloads(wname, causal, deterministic):
    """B4 H16 L4096 and B1 H32 L32768 (d = 128) on CTA pairs: sampled dQ rows
    and dK/dV rows over the whole sequence against the oracle on one head."""
    w = getattr(inputs, wname)
    t = inputs.make(w)
    dq, dk, dv = _grads(t, causal, w.scale, deterministic)
    head = [5]
    bsel = [w.B - 1]
    sub = {n: t[n][bsel] for n in ("q", "k", "v", "do")}
    qrows, krows = _rows(w.L, 12, 3), _rows(w.L, 12, 4)
    rq, rk, rv = oracle_bwd_subset(sub, w.scale, causal, heads=head, qrows=qrows, krows=krows)
    what = f"pair {w.name} causal={causal} det={deterministic}"
    assert_grad_close(to64(dq[bsel][:, qrows][:, :, head]), rq[:, qrows], f"{what} dQ")
    assert_grad_close(to64(dk[bsel][:, krows][:, :, head]), rk[:, krows], f"{what} dK")
    assert_grad_close(to64(dv[bsel][:, krows][:, :, head]), rv[:, krows], f"{what} dV")


@pytest.mark.parametrize("deterministic", [False, True])
def test_pair_workload_grouped(deterministic):
    """B2 H16 over 2 key/value heads, L8192 d128, causal, spiky K, on CTA pairs:
    dQ rows of query heads 3 and 12 against the oracle with their key/value
    heads; dK/dV rows of key/value head 1 against the oracle on its whole group."""
    import oracle
    w = inputs.HDSWEEP.with_(name="b2h16kv2l8192d128", hkv=2)
    t = inputs.make(w)
    dq, dk, dv = _grads(t, True, w.scale, deterministic)
    G = w.H // w.H_kv
    bsel = [0, w.B - 1]
    qrows, krows = _rows(w.L, 12, 5), _rows(w.L, 8, 6)
    qh = [3, 12]
    sub = {n: to64(t[n][bsel][:, :, qh]) for n in ("q", "do")}
    sub.update({n: to64(t[n][bsel][:, :, [h // G for h in qh]]) for n in ("k", "v")})
    rq, _, _ = oracle.bwd(sub["q"], sub["k"], sub["v"], sub["do"], w.scale, True, qrows=qrows, krows=[])
    assert_grad_close(to64(dq[bsel][:, qrows][:, :, qh]), rq[:, qrows], f"pair grouped workload det={deterministic} dQ")
    kh = 1
    grp = list(range(kh * G, kh * G + G))
    full = {n: to64(t[n][bsel][:, :, grp]) for n in ("q", "do")}
    full.update({n: to64(t[n][bsel][:, :, [kh]]) for n in ("k", "v")})
    _, rk, rv = oracle.bwd(full["q"], full["k"], full["v"], full["do"], w.scale, True, qrows=[], krows=krows)
    assert_grad_close(to64(dk[bsel][:, krows][:, :, [kh]]), rk[:, krows], f"pair grouped workload det={deterministic} dK")
    assert_grad_close(to64(dv[bsel][:, krows][:, :, [kh]]), rv[:, krows], f"pair grouped workload det={deterministic} dV")


@pytest.mark.parametrize("deterministic", [False, True])
def test_pair_workload_d64(deterministic):
    """B2 H16 L8192 d64, causal, spiky K, on CTA pairs (64-byte-swizzled column
    halves): sampled dQ rows and dK/dV rows over the whole sequence against the
    oracle on one head of each batch entry."""
    w = inputs.HDSWEEP.with_(d=64)
    t = inputs.make(w)
    dq, dk, dv = _grads(t, True, w.scale, deterministic)
    head = [9]
    qrows, krows = _rows(w.L, 12, 7), _rows(w.L, 12, 8)
    what = f"pair {w.name} det={deterministic}"
    for b in range(w.B):
        sub = {n: t[n][[b]] for n in ("q", "k", "v", "do")}
        rq, rk, rv = oracle_bwd_subset(sub, w.scale, True, heads=head, qrows=qrows, krows=krows)
        assert_grad_close(to64(dq[[b]][:, qrows][:, :, head]), rq[:, qrows], f"{what} b={b} dQ")
        assert_grad_close(to64(dk[[b]][:, krows][:, :, head]), rk[:, krows], f"{what} b={b} dK")
        assert_grad_close(to64(dv[[b]][:, krows][:, :, head]), rv[:, krows], f"{what} b={b} dV")
