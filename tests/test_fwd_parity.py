"""Forward parity: CUDA path (through the C ABI) vs the fp64 oracle.

Small problems are compared element by element over every output; the
workload shapes are compared on sampled rows of a subset of heads, in the
launch configuration the benchmark uses. Edge cases: ragged lengths that are
not multiples of the 128-row tiles, a single key, more queries than keys with
a causal mask (rows that see no key), empty batches, packed variable lengths.
"""
import numpy as np
import pytest
import torch

from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_fwd_close, oracle_fwd_subset, to64

pytestmark = pytest.mark.gpu


def run_dense(t, causal, scale):
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale)
    binding.check_status()
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_workload_full(causal):
    w = inputs.TINY
    t = inputs.make(w)
    o, lse = run_dense(t, causal, w.scale)
    o_ref, lse_ref = oracle_fwd_subset(t, w.scale, causal, heads=list(range(w.H)))
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, f"tiny causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 192, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [1, 77, 128, 129, 300, 513])
def test_ragged_lengths_full(L, causal, d):
    t = inputs.small(B=2, H=3, L=L, d=d, seed=7)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    o, lse = run_dense(t, causal, scale)
    o_ref, lse_ref = oracle_fwd_subset(t, scale, causal, heads=[0, 1, 2])
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, f"L={L} causal={causal} d={d}")


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(200, 77), (77, 300), (256, 1), (1, 256), (384, 129)])
def test_rectangular(Lq, Lk, causal, d):
    t = inputs.small(B=2, H=2, L=Lq, Lk=Lk, d=d, seed=8)
    scale = float(np.float32(0.088))
    o, lse = run_dense(t, causal, scale)
    o_ref, lse_ref = oracle_fwd_subset(t, scale, causal, heads=[0, 1])
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, f"Lq={Lq} Lk={Lk} causal={causal} d={d}")


@pytest.mark.parametrize("d", [64, 192])
def test_large_scores_and_rescaling(d):
    """Scores far larger than the rescale threshold, growing along the keys."""
    t = inputs.small(B=1, H=2, L=640, d=d, seed=9)
    ramp = torch.linspace(0.2, 6.0, 640).view(1, 640, 1, 1)
    t["k"] = (t["k"].float() * ramp).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = run_dense(t, causal, 0.5)
        o_ref, lse_ref = oracle_fwd_subset(t, 0.5, causal, heads=[0, 1])
        assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, f"spiky causal={causal} d={d}")


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_small_full(causal, d):
    lens = [1, 128, 200, 513, 77, 256]
    cu = inputs.cu_seqlens(lens)
    T, H = int(cu[-1]), 3
    g = torch.Generator("cpu").manual_seed(11)
    t = {n: torch.randn(T, H, d, generator=g).to(torch.bfloat16) for n in ("q", "k", "v")}
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o, lse = binding.forward(q, k, v, causal=causal, scale=0.1, cu_seqlens=cu.cuda())
    binding.check_status()
    o_ref, lse_ref = oracle_fwd_subset(t, 0.1, causal, heads=[0, 1, 2], cu=cu.numpy())
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, f"varlen causal={causal} d={d}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [1, 77, 128, 129, 300, 513])
def test_value_head_dim_192_128(L, causal):
    """q/k head dim 192 with v (and O) head dim 128 (attn_fwd_hdim)."""
    t = inputs.small(B=2, H=3, L=L, d=192, dv=128, seed=31)
    scale = float(np.float32(1.0 / np.sqrt(192)))
    o, lse = run_dense(t, causal, scale)
    assert o.shape == (2, L, 3, 128)
    o_ref, lse_ref = oracle_fwd_subset(t, scale, causal, heads=[0, 1, 2])
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, f"d192/dv128 L={L} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_value_head_dim_rectangular_and_varlen(causal):
    t = inputs.small(B=2, H=2, L=200, Lk=77, d=192, dv=128, seed=32)
    o, lse = run_dense(t, causal, 0.07)
    o_ref, lse_ref = oracle_fwd_subset(t, 0.07, causal, heads=[0, 1])
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, f"d192/dv128 Lq=200 Lk=77 causal={causal}")
    lens = [1, 128, 200, 513, 77, 256]
    cu = inputs.cu_seqlens(lens)
    T = int(cu[-1])
    g = torch.Generator("cpu").manual_seed(33)
    tv = {"q": torch.randn(T, 2, 192, generator=g).to(torch.bfloat16),
          "k": torch.randn(T, 2, 192, generator=g).to(torch.bfloat16),
          "v": torch.randn(T, 2, 128, generator=g).to(torch.bfloat16)}
    q, k, v = (tv[n].cuda() for n in ("q", "k", "v"))
    o, lse = binding.forward(q, k, v, causal=causal, scale=0.07, cu_seqlens=cu.cuda())
    binding.check_status()
    o_ref, lse_ref = oracle_fwd_subset(tv, 0.07, causal, heads=[0, 1], cu=cu.numpy())
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, f"d192/dv128 varlen causal={causal}")


def test_empty_batch_is_a_no_op():
    q = torch.empty(0, 128, 2, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = binding.forward(q, q, q, causal=True)
    binding.check_status()
    assert o.shape == q.shape


@pytest.mark.parametrize("d", [128, 192])
def test_repeated_calls_are_identical(d):
    t = inputs.small(B=1, H=2, L=700, d=d, seed=12)
    o1, l1 = run_dense(t, True, 0.09)
    o2, l2 = run_dense(t, True, 0.09)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------------------ workload shapes, sampled rows

def _sample_rows(L, n=24, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(L, size=min(n, L), replace=False).tolist())
    rows.update([0, 1, 127, 128, L - 1])
    return sorted(r for r in rows if 0 <= r < L)


def _workload_check(w, causal, heads):
    t = inputs.make(w, with_grad=False)
    o, lse = run_dense(t, causal, w.scale)
    rows = _sample_rows(w.L, seed=w.seed)
    bsel = sorted({0, w.B - 1})   # first and last batch entries
    sub = {n: t[n][bsel] for n in ("q", "k", "v")}
    o_ref, lse_ref = oracle_fwd_subset(sub, w.scale, causal, heads=heads, rows=rows)
    og = to64(o[bsel][:, rows][:, :, heads])
    lg = to64(lse[bsel][:, heads][:, :, rows])
    assert_fwd_close(og, lg, o_ref[:, rows], lse_ref[:, :, rows], f"{w.name} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_workload_b4h16l4096(causal):
    _workload_check(inputs.MHA4K, causal, heads=[0, 15])


@pytest.mark.parametrize("d", [64, 128, 192, 256])
def test_workload_hdsweep(d):
    _workload_check(inputs.HDSWEEP.with_(d=d), True, heads=[3])


def test_workload_hdsweep_value_head_dim():
    """B2 H16 L8192, q/k head dim 192, v head dim 128, causal, spiky K."""
    _workload_check(inputs.HDSWEEP.with_(d=192, dv=128), True, heads=[3])


@pytest.mark.parametrize("causal", [False, True])
def test_workload_long(causal):
    _workload_check(inputs.LONG, causal, heads=[7])


def test_workload_varlen():
    w = inputs.VARLEN
    t = inputs.make(w, with_grad=False)
    cu = t["cu_seqlens"]
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, cu_seqlens=cu.cuda())
    binding.check_status()
    lens = np.diff(cu.numpy())
    # shortest and longest sequence plus two others, two heads, sampled rows
    order = np.argsort(lens)
    for b in [int(order[0]), int(order[-1]), 5, 17]:
        a, L = int(cu[b]), int(lens[b])
        sub = {n: t[n][a:a + L].unsqueeze(0) for n in ("q", "k", "v")}
        rows = _sample_rows(L, n=12, seed=b)
        o_ref, lse_ref = oracle_fwd_subset(sub, w.scale, True, heads=[0, 9], rows=rows)
        og = to64(o[a:a + L][rows][:, [0, 9]])[None]
        lg = to64(lse[[0, 9]][:, a:a + L][:, rows])[None]
        assert_fwd_close(og, lg, o_ref[:, rows], lse_ref[:, :, rows], f"varlen seq {b} (L={L})")


# ------------------------------------------------------------------ partial exp2 emulation

class _exp2_emulation:
    """Set the forward's exp2 emulation for head dim d for the duration of a block."""

    def __init__(self, d, every):
        self.d, self.every = d, every

    def __enter__(self):
        self.prev = binding.attn_set_exp2_emulation(self.d, self.every)
        assert self.prev >= 0, binding.last_error()

    def __exit__(self, *exc):
        binding.attn_set_exp2_emulation(self.d, self.prev)
        return False


@pytest.mark.parametrize("every", [4, 8])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [77, 300, 640])
def test_exp2_emulation_full(L, causal, d, every):
    """The kernels with one column pair in 4 or 8 exponentiated by the FMA
    polynomial (FlashAttention-4 paper, Section 3.1.3): every element against
    the oracle, with growing scores so that rescaling runs too; and against the
    MUFU-only kernel, from which P differs by at most one bf16 ulp."""
    t = inputs.small(B=2, H=2, L=L, d=d, seed=12)
    ramp = torch.linspace(0.2, 4.0, L).view(1, L, 1, 1)
    t["k"] = (t["k"].float() * ramp).to(torch.bfloat16)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    with _exp2_emulation(d, 0):
        o_mufu, lse_mufu = run_dense(t, causal, scale)
    with _exp2_emulation(d, every):
        o, lse = run_dense(t, causal, scale)
    o_ref, lse_ref = oracle_fwd_subset(t, scale, causal, heads=[0, 1])
    what = f"poly 1/{every} L={L} causal={causal} d={d}"
    assert_fwd_close(to64(o), to64(lse), o_ref, lse_ref, what)
    assert float((o.float() - o_mufu.float()).abs().max()) <= 2e-2, what
    assert float((lse - lse_mufu).abs().max()) <= 1e-3, what


@pytest.mark.parametrize("every", [4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_exp2_emulation_workload(d, every):
    """B2 H16 L8192 causal with spiky K (the head-dim sweep workload), sampled rows."""
    w = inputs.HDSWEEP.with_(d=d)
    t = inputs.make(w)
    with _exp2_emulation(d, every):
        o, lse = run_dense(t, True, w.scale)
    rows = sorted({0, 1, 127, 128, 255, 256, 4095, 4096, w.L - 129, w.L - 1} |
                  set(np.random.default_rng(5).choice(w.L, 12, replace=False).tolist()))
    bsel = [0, w.B - 1]
    sub = {n: t[n][bsel] for n in ("q", "k", "v")}
    o_ref, lse_ref = oracle_fwd_subset(sub, w.scale, True, heads=[5], rows=rows)
    assert_fwd_close(to64(o[bsel][:, rows][:, :, [5]]), to64(lse[bsel][:, [5]][:, :, rows]),
                     o_ref[:, rows], lse_ref[:, :, rows], f"{w.name} poly 1/{every}")
