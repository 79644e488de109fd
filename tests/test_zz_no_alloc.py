"""attn_bwd_noalloc: the backward pass for callers that cannot allocate.

Some callers cannot give the library device memory of its own: code running
inside a framework or serving runtime that owns the whole device memory pool
and forbids allocations outside its own planner, or a plugin that only
receives its input and output pointers. attn_bwd_noalloc serves them with a
fixed scratch array built into the library instead of a workspace argument.

These tests call it through the C ABI, twice in a row on the same shared
scratch array (which keeps the previous call's contents, so the second call
checks that each call clears what it needs), and compare each call's
gradients
  * with those of attn_bwd, which takes a caller workspace (within the
    parity tests' tolerance; bit for bit in the deterministic mode, which runs
    the same kernels in the same order), and
  * with the fp64 oracle on every element.
The deterministic mode keeps its dQ semaphores in the scratch array, packed
sequences their longest-first sequence map: both have cases of their own.
This file is collected last on purpose, and also passes on its own.
"""
import numpy as np
import pytest
import torch

from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_grad_close, oracle_bwd_subset, to64

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 64 * 1024 * 1024   # ATTN_NOALLOC_SCRATCH_BYTES in include/attn.h


def _dense(B, H, L, d, seed):
    t = inputs.small(B=B, H=H, L=L, d=d, seed=seed)
    return t, None


def _packed(lens, H, d, seed):
    cu = inputs.cu_seqlens(lens)
    g = torch.Generator("cpu").manual_seed(seed)
    T = int(cu[-1])
    t = {n: torch.randn(T, H, d, generator=g).to(torch.bfloat16) for n in ("q", "k", "v", "do")}
    return t, cu


CASES = {
    "dense_causal_d128": (lambda: _dense(1, 4, 1000, 128, 31), True),
    "dense_d64": (lambda: _dense(2, 3, 777, 64, 32), False),
    "packed_causal_d128": (lambda: _packed([1, 128, 200, 513, 77, 256], 2, 128, 33), True),
    "packed_d64": (lambda: _packed([300, 5, 129, 640], 3, 64, 34), False),
}


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_workspace_entry_point_and_oracle(case, deterministic):
    make, causal = CASES[case]
    t, cu = make()
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    cud = cu.cuda() if cu is not None else None
    if cu is None:
        B, L, H, d = q.shape
    else:
        B, (L, H, d) = len(cu) - 1, q.shape
    scale = 1.0 / d ** 0.5
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale, cu_seqlens=cud)
    ref = binding.backward(q, k, v, o, lse, do, causal=causal, scale=scale, cu_seqlens=cud,
                           deterministic=bool(deterministic))
    binding.check_status()
    assert binding.attn_bwd_workspace_size(B, H, L, L, d, causal, deterministic) <= NOALLOC_BYTES
    heads = list(range(H))
    rq, rk, rv = oracle_bwd_subset(t, scale, causal, heads=heads, cu=None if cu is None else cu.numpy())
    first = None
    for call in range(2):
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
        rc = binding.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, B, H, L, L, d, scale, causal, cud,
                                      deterministic)
        assert rc == 0, binding.last_error()
        binding.check_status()
        what = f"noalloc {case} det={deterministic} call {call}"
        for name, got, want, orc in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref, (rq, rk, rv)):
            assert_grad_close(to64(got), to64(want), f"{what} {name} vs attn_bwd")
            assert_grad_close(to64(got), orc, f"{what} {name} vs oracle")
            if deterministic:
                assert torch.equal(got, want), f"{what} {name}: not bit-identical to attn_bwd"
        if first is None:
            first = (dq, dk, dv)
        elif deterministic:
            for a, b in zip(first, (dq, dk, dv)):
                assert torch.equal(a, b), f"{what}: two deterministic calls differ"


def test_noalloc_rejects_problems_beyond_its_scratch():
    B, H, L, d = 4, 16, 4096, 128   # needs ~128 MiB of scratch
    assert binding.attn_bwd_workspace_size(B, H, L, L, d, 1, 0) > NOALLOC_BYTES
    dummy = 1 << 20                  # never dereferenced: the size check fails first
    rc = binding.attn_bwd_noalloc(*([dummy] * 9), B, H, L, L, d, 0.088, 1, None, 0)
    assert rc == binding.ATTN_ERR_WORKSPACE
    assert "scratch" in binding.last_error()
