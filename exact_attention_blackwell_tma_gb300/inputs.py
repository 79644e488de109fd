"""Seeded synthetic inputs for the attention workloads.

This module is shared by the CUDA path's tests/benchmark and by the CPU
oracle's tests. It holds no attention arithmetic: it only draws numbers.

Recipe (the pages measure on synthetic shapes only -- FlashAttention-4 paper,
Section 5, Figs. 4-8 sweep sequence length and head dim):
  * every tensor is drawn i.i.d. N(0, 1) in fp32 from ``torch.Generator('cpu')``
    and rounded to bf16 (round-to-nearest-even); the same bf16 bits go to the
    GPU and (widened exactly) to the oracle;
  * a workload with seed ``s`` draws Q, K, V, dO from seeds ``10*s + 0..3``;
  * the head-dim sweep multiplies K by 4 on a random 5% of sequence positions
    (seed ``10*s + 4``; the same positions for every head of a batch entry) so
    that the running row maximum jumps and conditional rescaling is exercised;
  * the variable-length batch draws its sequence lengths uniformly from
    ``[lo, hi]`` (seed ``10*s + 5``) and packs the sequences back to back;
  * grouped heads: K and V (and the spikes) are drawn with ``hkv`` heads;
  * a batch with key lengths of their own (``lengths_k``) packs K and V by
    those lengths; the prefill/decode mix draws (seed ``10*s + 6``) half its
    sequences as prefill (queries = keys, uniform in ``[lo, hi]``) and half
    as decode steps (1 to 16 queries against a key cache uniform in
    ``[lo_k, hi_k]``), in a shuffled order.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem shape. ``lengths`` set => packed variable-length."""
    name: str
    B: int
    H: int
    L: int
    d: int
    causal: bool
    seed: int
    kspike_frac: float = 0.0          # fraction of positions whose K rows are scaled
    kspike: float = 4.0
    lengths: Optional[tuple] = None   # varlen: per-sequence lengths
    dv: Optional[int] = None          # head dim of v (and dO); None: the same as q and k
    hkv: Optional[int] = None         # key/value heads (grouped heads); None: H
    lengths_k: Optional[tuple] = None # varlen: per-sequence key lengths; None: the query lengths
    window: tuple = (-1, -1)          # local window (left, right); -1: open side
    block_pattern: Optional[tuple] = None   # ("local_strided", local, stride): block mask pattern

    @property
    def scale(self) -> float:
        """1/sqrt(d), rounded to fp32 (the C ABI takes a 32-bit float)."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    @property
    def d_v(self) -> int:
        return self.d if self.dv is None else self.dv

    @property
    def H_kv(self) -> int:
        return self.H if self.hkv is None else self.hkv

    @property
    def varlen(self) -> bool:
        return self.lengths is not None

    @property
    def total(self) -> int:
        return sum(self.lengths) if self.varlen else self.B * self.L

    @property
    def keys(self) -> tuple:
        """Per-sequence key lengths of a varlen batch."""
        return self.lengths if self.lengths_k is None else self.lengths_k

    @property
    def total_k(self) -> int:
        return sum(self.keys) if self.varlen else self.B * self.L

    def pairs(self) -> int:
        """Number of unmasked (query, key) pairs summed over batch and heads
        (causal: bottom-right aligned, j <= i + Lk - Lq; a local window keeps
        i + Lk - Lq - left <= j <= i + Lk - Lq + right)."""
        wl, wr = self.window
        if self.causal:
            wr = 0

        def per_seq(lq, lk):
            if wl < 0 and wr < 0:
                return lq * lk
            i = torch.arange(lq, dtype=torch.int64)
            lo = (i + (lk - lq) - wl).clamp(min=0) if wl >= 0 else torch.zeros_like(i)
            hi = (i + (lk - lq) + wr + 1).clamp(max=lk) if wr >= 0 else torch.full_like(i, lk)
            return int((hi - lo).clamp(min=0).sum())
        if self.varlen:
            return self.H * sum(per_seq(a, b) for a, b in zip(self.lengths, self.keys))
        if self.block_pattern is not None:
            return self.B * self.H * _pairs_in_blocks(block_mask(self)[0], self.L, self.L, wl, wr)
        return self.B * self.H * per_seq(self.L, self.L)

    def fwd_flops(self) -> int:
        """Algorithmic forward FLOPs: 2*d (S = Q K^T) + 2*d_v (O = P V) per unmasked pair."""
        return 2 * (self.d + self.d_v) * self.pairs()

    def bwd_flops(self) -> int:
        """Algorithmic backward FLOPs: five GEMMs per unmasked pair -- S and dK, dQ
        over d, dP and dV over d_v: 2 * (3 d + 2 d_v) (2.5x the forward when d_v = d)."""
        return 2 * (3 * self.d + 2 * self.d_v) * self.pairs()

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def block_mask(w: Workload):
    """The workload's block mask, uint8 [1, ceil(L/128), ceil(L/128)], from its
    pattern: ("local_strided", a, s) keeps, for query block q, key blocks
    q-a+1 .. q and every key block k with k % s == s - 1."""
    kind, a, st = w.block_pattern
    assert kind == "local_strided"
    n = -(-w.L // 128)
    qb = torch.arange(n)[:, None]
    kb = torch.arange(n)[None, :]
    keep = ((qb - kb >= 0) & (qb - kb < a)) | (kb % st == st - 1)
    return keep.to(torch.uint8)[None]


def _pairs_in_blocks(mask2d, lq, lk, wl, wr) -> int:
    """Pairs a block mask keeps inside the band (for the FLOP count)."""
    i = torch.arange(lq, dtype=torch.int64)
    lo = (i + (lk - lq) - wl).clamp(min=0) if wl >= 0 else torch.zeros_like(i)
    hi = (i + (lk - lq) + wr + 1).clamp(max=lk) if wr >= 0 else torch.full_like(i, lk)
    rows = mask2d[(i // 128)].to(torch.bool)                        # [lq, nkb]
    k0 = torch.arange(mask2d.shape[1], dtype=torch.int64)[None, :] * 128
    cnt = (torch.minimum(hi[:, None], (k0 + 128).clamp(max=lk)) - torch.maximum(lo[:, None], k0)).clamp(min=0)
    return int((cnt * rows).sum())


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    g = torch.Generator("cpu").manual_seed(10 * seed + 5)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g))


def prefill_decode_lengths(n: int, lo: int, hi: int, lo_k: int, hi_k: int, seed: int):
    """(query lengths, key lengths) of n sequences, half prefill, half decode."""
    g = torch.Generator("cpu").manual_seed(10 * seed + 6)
    lq, lk = [], []
    for i in range(n):
        if i < n // 2:
            L = int(torch.randint(lo, hi + 1, (1,), generator=g))
            lq.append(L)
            lk.append(L)
        else:
            lq.append(int(torch.randint(1, 17, (1,), generator=g)))
            lk.append(int(torch.randint(lo_k, hi_k + 1, (1,), generator=g)))
    perm = torch.randperm(n, generator=g).tolist()
    return tuple(lq[i] for i in perm), tuple(lk[i] for i in perm)


def cu_seqlens(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


# The five workloads. Names describe the shape.
TINY = Workload("tiny_b1h2l128d64", B=1, H=2, L=128, d=64, causal=False, seed=1)
MHA4K = Workload("b4h16l4096d128", B=4, H=16, L=4096, d=128, causal=True, seed=2)
HDSWEEP = Workload("b2h16l8192", B=2, H=16, L=8192, d=128, causal=True, seed=3, kspike_frac=0.05)
VARLEN = Workload("varlen32_h16d128", B=32, H=16, L=16384, d=128, causal=True, seed=4,
                  lengths=varlen_lengths(32, 256, 16384, 4))
LONG = Workload("b1h32l32768d128", B=1, H=32, L=32768, d=128, causal=True, seed=5)
_PD_Q, _PD_K = prefill_decode_lengths(32, 256, 8192, 1024, 16384, 6)
PREFILL_DECODE = Workload("mix32_prefill_decode_h16kv4d128", B=32, H=16, L=16384, d=128, causal=True, seed=6,
                          lengths=_PD_Q, lengths_k=_PD_K, hkv=4)


def _randn(shape, seed: int) -> torch.Tensor:
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32)


def make(w: Workload, with_grad: bool = True) -> dict:
    """Draw q, k, v (and dO) for a workload as CPU bf16 tensors.

    Dense layout ``[B, L, H, d]``; varlen ``[T, H, d]`` plus ``cu_seqlens``.
    """
    shape = (w.total, w.H, w.d) if w.varlen else (w.B, w.L, w.H, w.d)
    kshape = (w.total_k, w.H_kv, w.d) if w.varlen else (w.B, w.L, w.H_kv, w.d)
    q = _randn(shape, 10 * w.seed + 0)
    k = _randn(kshape, 10 * w.seed + 1)
    v = _randn(kshape[:-1] + (w.d_v,), 10 * w.seed + 2)
    if w.kspike_frac > 0:
        g = torch.Generator("cpu").manual_seed(10 * w.seed + 4)
        n = max(1, int(round(w.kspike_frac * w.L)))
        if w.varlen:
            raise ValueError("K spikes are defined for dense workloads only")
        for b in range(w.B):
            pos = torch.randperm(w.L, generator=g)[:n]
            k[b, pos] *= w.kspike
    out = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    if with_grad:
        out["do"] = _randn(shape[:-1] + (w.d_v,), 10 * w.seed + 3).to(torch.bfloat16)
    if w.varlen:
        out["cu_seqlens"] = cu_seqlens(w.lengths)
        if w.lengths_k is not None:
            out["cu_seqlens_k"] = cu_seqlens(w.lengths_k)
    return out


def small(B=1, H=2, L=128, d=64, causal=False, seed=1, Lk=None, dv=None, Hkv=None) -> dict:
    """Small dense problem with possibly different query and key lengths (a
    head dim of its own for v and dO, and fewer key/value heads)."""
    Lk = L if Lk is None else Lk
    dv = d if dv is None else dv
    Hkv = H if Hkv is None else Hkv
    return {
        "q": _randn((B, L, H, d), 10 * seed + 0).to(torch.bfloat16),
        "k": _randn((B, Lk, Hkv, d), 10 * seed + 1).to(torch.bfloat16),
        "v": _randn((B, Lk, Hkv, dv), 10 * seed + 2).to(torch.bfloat16),
        "do": _randn((B, L, H, dv), 10 * seed + 3).to(torch.bfloat16),
    }
