"""Backward parity: dQ, dK, dV from the CUDA path (through the C ABI) vs the
fp64 oracle, plus the deterministic mode's bit-reproducibility.

The backward consumes the forward's O and LSE from the CUDA path (as a user
would); the oracle recomputes everything from q, k, v, dO by the definition.
Small problems are compared over every element; the workload shapes on
sampled query rows (dQ) and key rows (dK, dV) drawn over the whole sequence,
in the default and the deterministic mode, and over whole tensors through two
identities that hold at any size: sum_j dV_j = sum_i dO_i and sum_j dK_j = 0
(rows of P sum to one; rows of dS sum to zero).
"""
import numpy as np
import pytest
import torch

from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_grad_close, oracle_bwd_subset, rel_l2, to64

pytestmark = pytest.mark.gpu


def run_dense(t, causal, scale, deterministic=False):
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = binding.backward(q, k, v, o, lse, do, causal=causal, scale=scale, deterministic=deterministic)
    binding.check_status()
    return dq, dk, dv


def check_all(t, causal, scale, heads, what, deterministic=False):
    dq, dk, dv = run_dense(t, causal, scale, deterministic)
    rq, rk, rv = oracle_bwd_subset(t, scale, causal, heads=heads)
    assert_grad_close(to64(dq[:, :, heads]), rq, f"{what} dQ")
    assert_grad_close(to64(dk[:, :, heads]), rk, f"{what} dK")
    assert_grad_close(to64(dv[:, :, heads]), rv, f"{what} dV")


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_tiny_workload_full(causal, deterministic):
    w = inputs.TINY
    check_all(inputs.make(w), causal, w.scale, list(range(w.H)), f"tiny causal={causal}", deterministic)


@pytest.mark.parametrize("d", [64, 128, 192, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [1, 77, 129, 300])
def test_ragged_lengths_full(L, causal, d):
    t = inputs.small(B=2, H=2, L=L, d=d, seed=21)
    check_all(t, causal, float(np.float32(1 / np.sqrt(d))), [0, 1], f"L={L} causal={causal} d={d}")


@pytest.mark.parametrize("d", [64, 192])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(200, 77), (77, 300), (384, 129)])
def test_rectangular(Lq, Lk, causal, d):
    t = inputs.small(B=1, H=2, L=Lq, Lk=Lk, d=d, seed=22)
    check_all(t, causal, 0.125, [0, 1], f"Lq={Lq} Lk={Lk} causal={causal} d={d}")


@pytest.mark.parametrize("d", [128, 192, 256])
@pytest.mark.parametrize("deterministic", [False, True])
def test_varlen_small_full(deterministic, d):
    lens = [1, 128, 200, 513, 77, 256]
    cu = inputs.cu_seqlens(lens)
    T, H = int(cu[-1]), 2
    g = torch.Generator("cpu").manual_seed(23)
    t = {n: torch.randn(T, H, d, generator=g).to(torch.bfloat16) for n in ("q", "k", "v", "do")}
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    cud = cu.cuda()
    o, lse = binding.forward(q, k, v, causal=True, scale=0.1, cu_seqlens=cud)
    dq, dk, dv = binding.backward(q, k, v, o, lse, do, causal=True, scale=0.1, cu_seqlens=cud,
                                  deterministic=deterministic)
    binding.check_status()
    rq, rk, rv = oracle_bwd_subset(t, 0.1, True, heads=[0, 1], cu=cu.numpy())
    assert_grad_close(to64(dq), rq, f"varlen d={d} dQ")
    assert_grad_close(to64(dk), rk, f"varlen d={d} dK")
    assert_grad_close(to64(dv), rv, f"varlen d={d} dV")


@pytest.mark.parametrize("d", [128, 192])
@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_is_bit_identical(causal, d):
    t = inputs.small(B=2, H=4, L=1024, d=d, seed=24)
    ref = run_dense(t, causal, 0.088, deterministic=True)
    for _ in range(4):
        again = run_dense(t, causal, 0.088, deterministic=True)
        for a, b in zip(ref, again):
            assert torch.equal(a, b)


# ------------------------------------------------------------------ d_qk = 192, d_v = 128

@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [1, 77, 129, 300])
def test_value_head_dim_192_128(L, causal, deterministic):
    """q/k head dim 192, v (dO, dV) head dim 128: every element of dQ, dK, dV."""
    t = inputs.small(B=2, H=2, L=L, d=192, dv=128, seed=25)
    check_all(t, causal, float(np.float32(1 / np.sqrt(192))), [0, 1], f"d192/dv128 L={L} causal={causal}",
              deterministic)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(200, 77), (77, 300)])
def test_value_head_dim_rectangular(Lq, Lk, causal):
    t = inputs.small(B=1, H=2, L=Lq, Lk=Lk, d=192, dv=128, seed=26)
    check_all(t, causal, 0.07, [0, 1], f"d192/dv128 Lq={Lq} Lk={Lk} causal={causal}")


@pytest.mark.parametrize("deterministic", [False, True])
def test_value_head_dim_grouped_varlen(deterministic):
    """d192/dv128 with grouped heads (split over tiles: partial dK slots 192
    wide, dV slots 128 wide) and packed sequences with key offsets of their own."""
    lq, lk = [1, 128, 200, 513, 0, 300], [300, 1, 200, 129, 77, 256]
    cu, cuk = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    g = torch.Generator("cpu").manual_seed(27)
    Tq, Tk, H, Hkv = int(cu[-1]), int(cuk[-1]), 4, 2
    t = {"q": torch.randn(Tq, H, 192, generator=g).to(torch.bfloat16),
         "k": torch.randn(Tk, Hkv, 192, generator=g).to(torch.bfloat16),
         "v": torch.randn(Tk, Hkv, 128, generator=g).to(torch.bfloat16),
         "do": torch.randn(Tq, H, 128, generator=g).to(torch.bfloat16)}
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    cq, ck = cu.cuda(), cuk.cuda()
    o, lse = binding.forward(q, k, v, causal=True, scale=0.07, cu_seqlens=cq, cu_seqlens_k=ck)
    dq, dk, dv = binding.backward(q, k, v, o, lse, do, causal=True, scale=0.07, cu_seqlens=cq, cu_seqlens_k=ck,
                                  deterministic=deterministic)
    binding.check_status()
    assert dv.shape == (Tk, Hkv, 128)
    import oracle
    rq, rk, rv = oracle.bwd(*(to64(t[n]) for n in ("q", "k", "v", "do")), 0.07, True, cu_seqlens=cu.numpy(),
                            cu_seqlens_k=cuk.numpy())
    assert_grad_close(to64(dq), rq, "d192/dv128 grouped varlen dQ")
    assert_grad_close(to64(dk), rk, "d192/dv128 grouped varlen dK")
    assert_grad_close(to64(dv), rv, "d192/dv128 grouped varlen dV")


def test_value_head_dim_deterministic_is_bit_identical():
    t = inputs.small(B=2, H=4, L=1024, d=192, dv=128, seed=28)
    ref = run_dense(t, True, 0.07, deterministic=True)
    for _ in range(3):
        again = run_dense(t, True, 0.07, deterministic=True)
        for a, b in zip(ref, again):
            assert torch.equal(a, b)


# ------------------------------------------------------------------ workload shapes

def _rows(L, n, seed):
    """n seeded rows of [0, L) plus both edges of the first block boundary and the last row."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(L, size=min(n, L), replace=False).tolist()) | {0, 127, 128, L - 1}
    return sorted(r for r in rows if 0 <= r < L)


def _identities(t, dk, dv, what):
    """sum_j dV_j = sum_i dO_i and sum_j dK_j = 0, per batch and head, over whole tensors."""
    sdv = dv.float().sum(dim=1)
    sdo = t["do"].cuda().float().sum(dim=1)
    e = rel_l2(sdv.double().cpu().numpy(), sdo.double().cpu().numpy())
    assert e < 2e-2, f"{what}: sum dV vs sum dO rel {e:.3e}"
    sdk = dk.float().sum(dim=1)
    scale = dk.float().pow(2).sum(dim=1).sqrt()
    ratio = float((sdk.norm() / scale.norm()).item())
    assert ratio < 5e-2, f"{what}: |sum dK| / |dK| = {ratio:.3e}"


def _workload_check(w, causal, heads, deterministic=False):
    t = inputs.make(w)
    dq, dk, dv = run_dense(t, causal, w.scale, deterministic)
    qrows = _rows(w.L, 16, w.seed)
    krows = _rows(w.L, 12, w.seed + 1)
    bsel = sorted({0, w.B - 1})   # first and last batch entries
    sub = {n: t[n][bsel] for n in ("q", "k", "v", "do")}
    rq, rk, rv = oracle_bwd_subset(sub, w.scale, causal, heads=heads, qrows=qrows, krows=krows)
    assert_grad_close(to64(dq[bsel][:, qrows][:, :, heads]), rq[:, qrows], f"{w.name} dQ")
    assert_grad_close(to64(dk[bsel][:, krows][:, :, heads]), rk[:, krows], f"{w.name} dK")
    assert_grad_close(to64(dv[bsel][:, krows][:, :, heads]), rv[:, krows], f"{w.name} dV")
    _identities(t, dk, dv, w.name)


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_workload_b4h16l4096(causal, deterministic):
    _workload_check(inputs.MHA4K, causal, heads=[0, 15], deterministic=deterministic)


@pytest.mark.parametrize("d", [64, 128, 192, 256])
def test_workload_hdsweep(d):
    _workload_check(inputs.HDSWEEP.with_(d=d), True, heads=[3])


@pytest.mark.parametrize("d", [64, 128])
def test_workload_hdsweep_deterministic(d):
    """B2 H16 L8192 causal, spiky K, deterministic mode: sampled rows against the
    oracle and two runs bit-identical (d = 64 runs the order with dQ and dS^T in
    tensor-memory columns of their own, issued from lane 0 in this mode)."""
    w = inputs.HDSWEEP.with_(d=d)
    _workload_check(w, True, heads=[3], deterministic=True)
    t = inputs.make(w)
    a = run_dense(t, True, w.scale, True)
    b = run_dense(t, True, w.scale, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_workload_hdsweep_value_head_dim():
    """B2 H16 L8192, q/k head dim 192, v head dim 128, causal, spiky K."""
    _workload_check(inputs.HDSWEEP.with_(d=192, dv=128), True, heads=[3])


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_workload_long(causal, deterministic):
    """B1 H32 L32768: dQ rows and dK/dV rows sampled over the whole sequence
    (key blocks 0 and 1 included: with a causal mask they see every query
    block, and in the deterministic mode they take the most semaphore turns),
    against the fp64 oracle on one head; deterministic runs also repeat bit
    for bit."""
    w = inputs.LONG
    t = inputs.make(w)
    got = run_dense(t, causal, w.scale, deterministic)
    if deterministic:
        again = run_dense(t, causal, w.scale, deterministic)
        for x, y in zip(got, again):
            assert torch.equal(x, y)
    dq, dk, dv = got
    heads = [7]
    qrows = _rows(w.L, 16, w.seed)
    krows = sorted(set(_rows(w.L, 12, w.seed + 1)) | {1, 64, 200, w.L // 2, w.L // 2 + 77})
    rq, rk, rv = oracle_bwd_subset(t, w.scale, causal, heads=heads, qrows=qrows, krows=krows)
    what = f"{w.name} causal={causal} det={deterministic}"
    assert_grad_close(to64(dq[:, qrows][:, :, heads]), rq[:, qrows], f"{what} dQ")
    assert_grad_close(to64(dk[:, krows][:, :, heads]), rk[:, krows], f"{what} dK")
    assert_grad_close(to64(dv[:, krows][:, :, heads]), rv[:, krows], f"{what} dV")
    _identities(t, dk, dv, what)


@pytest.mark.parametrize("deterministic", [False, True])
def test_workload_varlen(deterministic):
    w = inputs.VARLEN
    t = inputs.make(w)
    cu = t["cu_seqlens"]
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    cud = cu.cuda()
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, cu_seqlens=cud)
    dq, dk, dv = binding.backward(q, k, v, o, lse, do, causal=True, scale=w.scale, cu_seqlens=cud,
                                  deterministic=deterministic)
    binding.check_status()
    if deterministic:
        again = binding.backward(q, k, v, o, lse, do, causal=True, scale=w.scale, cu_seqlens=cud,
                                 deterministic=True)
        binding.check_status()
        for x, y in zip((dq, dk, dv), again):
            assert torch.equal(x, y)
    lens = np.diff(cu.numpy())
    order = np.argsort(lens)
    for b in [int(order[0]), int(order[-1]), 5]:
        a, L = int(cu[b]), int(lens[b])
        sub = {n: t[n][a:a + L].unsqueeze(0) for n in ("q", "k", "v", "do")}
        qrows = _rows(L, 10, b)
        # key rows over the whole sequence: the first ones see every query row
        krows = _rows(L, 8, b + 1)
        rq, rk, rv = oracle_bwd_subset(sub, w.scale, True, heads=[0, 9], qrows=qrows, krows=krows)
        what = f"varlen seq {b} det={deterministic}"
        assert_grad_close(to64(dq[a:a + L][qrows][:, [0, 9]])[None], rq[:, qrows], f"{what} dQ")
        assert_grad_close(to64(dk[a:a + L][krows][:, [0, 9]])[None], rk[:, krows], f"{what} dK")
        assert_grad_close(to64(dv[a:a + L][krows][:, [0, 9]])[None], rv[:, krows], f"{what} dV")
