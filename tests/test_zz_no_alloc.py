"""attn_bwd_noalloc: the backward pass for callers that cannot allocate.

Some callers cannot give the library device memory of its own: code running
inside a framework or serving runtime that owns the whole device memory pool
and forbids allocations outside its own planner, or a plugin that only
receives its input and output pointers. attn_bwd_noalloc serves them with a
fixed scratch array built into the library instead of a workspace argument.

These tests call it through the C ABI and compare its gradients with those of
attn_bwd (which takes a caller workspace), within the tolerance the parity
tests use, on two calls in a row: the scratch array keeps the previous call's
contents, so the second call checks that each call clears what it needs.
This file is collected last on purpose, and also passes on its own.
"""
import pytest
import torch

from exact_attention_blackwell_tma_gb300 import binding, inputs
from _util import assert_grad_close, to64

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 64 * 1024 * 1024   # ATTN_NOALLOC_SCRATCH_BYTES in include/attn.h


def _problem(B, H, L, d, seed):
    t = inputs.small(B=B, H=H, L=L, d=d, seed=seed)
    return {n: x.cuda() for n, x in t.items()}


@pytest.mark.parametrize("B,H,L,d,causal", [(1, 4, 1000, 128, True), (2, 3, 777, 64, False)])
def test_noalloc_matches_workspace_entry_point(B, H, L, d, causal):
    t = _problem(B, H, L, d, seed=31)
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    scale = 1.0 / d ** 0.5
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale)
    ref = binding.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    binding.check_status()
    assert binding.attn_bwd_workspace_size(B, H, L, L, d, causal, 0) <= NOALLOC_BYTES
    for call in range(2):
        dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
        rc = binding.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, B, H, L, L, d, scale, causal, None, 0)
        assert rc == 0, binding.last_error()
        binding.check_status()
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert_grad_close(to64(got), to64(want), f"noalloc call {call} {name}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    B, H, L, d = 4, 16, 4096, 128   # needs ~128 MiB of scratch
    assert binding.attn_bwd_workspace_size(B, H, L, L, d, 1, 0) > NOALLOC_BYTES
    dummy = 1 << 20                  # never dereferenced: the size check fails first
    rc = binding.attn_bwd_noalloc(*([dummy] * 9), B, H, L, L, d, 0.088, 1, None, 0)
    assert rc == binding.ATTN_ERR_WORKSPACE
    assert "scratch" in binding.last_error()
