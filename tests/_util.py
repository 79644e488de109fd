"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs, then compare.

Tolerances (bf16 inputs and outputs, fp32 accumulation):
  O and LSE: max |err| <= 2e-2 and mean |err| <= 2e-3;
  dQ, dK, dV: relative L2 error <= 2e-2 (per tensor, over the compared rows).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

O_MAX, O_MEAN = 2e-2, 2e-3
GRAD_REL_L2 = 2e-2
# Where the exact gradient is zero by construction -- a single visible key makes
# dS = 0, hence dQ = dK = 0 -- a relative error has no meaning. Such a tensor is
# recognised by its oracle RMS (zero up to fp64 rounding, below ZERO_RMS), and
# only then is the GPU's rounding noise judged absolutely: its RMS must stay
# below GRAD_REL_L2 * GRAD_RMS_FLOOR. Every other tensor gets the plain relative
# L2 error, however small its norm.
GRAD_RMS_FLOOR = 1e-3
ZERO_RMS = 1e-10


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def lse_errors(got: np.ndarray, ref: np.ndarray):
    """Max/mean abs error of LSE; -inf entries must agree exactly."""
    ninf_g, ninf_r = np.isneginf(got), np.isneginf(ref)
    assert np.array_equal(ninf_g, ninf_r), "rows with no visible key disagree"
    fin = ~ninf_r
    if not fin.any():
        return 0.0, 0.0
    d = np.abs(got[fin] - ref[fin])
    return float(d.max()), float(d.mean())


def assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite O"
    d = np.abs(o_gpu - o_ref)
    omax, omean = float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0
    lmax, lmean = lse_errors(lse_gpu, lse_ref)
    assert omax <= O_MAX and omean <= O_MEAN, f"{what}: O max {omax:.3e} mean {omean:.3e}"
    assert lmax <= O_MAX and lmean <= O_MEAN, f"{what}: LSE max {lmax:.3e} mean {lmean:.3e}"
    return omax, omean, lmax, lmean


def rel_l2(got: np.ndarray, ref: np.ndarray, floor_rms: float = 0.0) -> float:
    n = max(np.linalg.norm(ref), floor_rms * np.sqrt(ref.size), 1e-30)
    return float(np.linalg.norm(got - ref) / n)


def assert_grad_close(got, ref, what=""):
    assert np.isfinite(got).all(), f"{what}: non-finite gradient"
    if ref.size and np.sqrt(np.mean(ref * ref)) < ZERO_RMS:
        e = rel_l2(got, ref, GRAD_RMS_FLOOR)
        assert e <= GRAD_REL_L2, f"{what}: exact gradient is zero; RMS {e * GRAD_RMS_FLOOR:.3e} (absolute)"
        return e
    e = rel_l2(got, ref)
    assert e <= GRAD_REL_L2, f"{what}: rel L2 {e:.3e}"
    return e


def dense_inputs_on_gpu(t: dict):
    return {k: v.cuda() for k, v in t.items()}


def head_slice(t: torch.Tensor, heads, varlen: bool):
    """Select heads of a [B, L, H, d] (or [T, H, d]) tensor, as float64 numpy."""
    if varlen:
        return to64(t[:, heads])
    return to64(t[:, :, heads])


def oracle_fwd_subset(t: dict, scale, causal, heads, rows=None, cu=None):
    varlen = cu is not None
    q, k, v = (head_slice(t[n], heads, varlen) for n in ("q", "k", "v"))
    return oracle.fwd(q, k, v, scale, causal, cu_seqlens=cu, rows=rows)


def oracle_bwd_subset(t: dict, scale, causal, heads, qrows=None, krows=None, cu=None):
    varlen = cu is not None
    q, k, v, do = (head_slice(t[n], heads, varlen) for n in ("q", "k", "v", "do"))
    return oracle.bwd(q, k, v, do, scale, causal, cu_seqlens=cu, qrows=qrows, krows=krows)
