#!/usr/bin/env python
"""Throughput benchmark of the attention hot path on GB300.

A step is one pass of the whole path over one batch of synthetic input: for
each mask variant of the workload, the forward and the backward (preprocess,
main kernel, dQ conversion), called through the general entry points
attn_fwd_ex / attn_bwd_ex (attn_fwd_varlen / attn_bwd_varlen for the
prefill/decode mix). The default workload is the long-context one,
B=1, H=32, L=32768, d=128 (bf16), causal and non-causal: the largest
configuration of the five the parity tests cover. Throughput is algorithmic
FLOPs / time: forward 2*(d + d_v) per unmasked (query, key) pair, backward
2*(3d + 2d_v) (2.5x the forward when d_v = d).

Beside the step, the same run times two single calls with their own roofline
fraction: the causal forward at B=2, H=16, L=8192, d=128 (the workload whose
forward has a stated goal of 55% of the dense BF16 peak), and the
deterministic causal backward of the default workload.

  python bench.py [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0). Under torchrun each rank runs the same
workload on its own GPU (independent replicas, no collective on the data
path: weak scaling); the timed region is bracketed by a barrier and a device
synchronise, and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import copy
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from exact_attention_blackwell_tma_gb300 import binding, inputs  # noqa: E402

METRIC = "attention fwd/bwd TFLOPS (bf16, causal+non-causal) and % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"

WORKLOADS = {
    "b4h16l4096d128": (inputs.MHA4K, (True, False)),
    "b2h16l8192d128": (inputs.HDSWEEP, (True,)),
    "b2h16l8192d64": (inputs.HDSWEEP.with_(d=64), (True,)),
    "b2h16l8192d192": (inputs.HDSWEEP.with_(d=192), (True,)),
    "b2h16l8192d256": (inputs.HDSWEEP.with_(d=256), (True,)),
    # q/k head dim 192 with v head dim 128 (attn_fwd_ex / attn_bwd_ex)
    "b2h16l8192dqk192dv128": (inputs.HDSWEEP.with_(d=192, dv=128), (True,)),
    # causal with a local window of 4096 keys (attn_fwd_ex / attn_bwd_ex window bounds)
    "b2h16l8192d128_window4096": (inputs.HDSWEEP.with_(name="b2h16l8192d128_window4096", window=(4096, 0)), (True,)),
    # causal with a block mask: each query block keeps its 4 nearest key blocks and every 8th
    "b2h16l8192d128_blocksparse": (inputs.HDSWEEP.with_(name="b2h16l8192d128_blocksparse",
                                                        block_pattern=("local_strided", 4, 8)), (True,)),
    # grouped heads: 16 query heads over 2 key/value heads
    "b2h16kv2l8192d128": (inputs.HDSWEEP.with_(name="b2h16kv2l8192d128", hkv=2), (True,)),
    "varlen32_h16d128": (inputs.VARLEN, (True,)),
    # 16 prefill sequences (queries = keys) and 16 decode steps (1-16 queries
    # against a long key cache), 4 key/value heads (attn_fwd_varlen / attn_bwd_varlen)
    "mix32_prefill_decode_h16kv4d128": (inputs.PREFILL_DECODE, (True,)),
    "b1h32l32768d128": (inputs.LONG, (True, False)),
}
DEFAULT_WORKLOAD = "b1h32l32768d128"
# the causal forward at d = 128, L = 8192 must reach this fraction of the dense BF16 peak
TARGET_WORKLOAD, TARGET_FRAC = "b2h16l8192d128", 0.55
L2_BYTES = 129 * 1024 * 1024


def kinds_of(w):
    """The calls a step makes: the forward and the backward."""
    return ("fwd", "bwd")

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a
# workload's dominant kernel, from the ncu capture summarised in the named
# profile. It holds only for the kernel sources it was taken on: their SHA-256
# is checked at run time and the field is reported as null after any change.
NCU_TRAFFIC = {
    ("b1h32l32768d128", "bwd", False): {
        "bytes": 8728.203e6 + 4564.870e6,
        "profile": "profiles/bwd_kernel_b1h32l32768d128_traffic.md",
        "sources": {
            "exact_attention_blackwell_tma_gb300/csrc/bwd.cu":
                "60bc2511e502cc06be6d193c1279504a2fdce162ce618fc40e08004425c032ba",
            "exact_attention_blackwell_tma_gb300/csrc/ptx.cuh":
                "3c0283284f2342dd722773b9195bbfdc67274aa16994dbb143983c848529bf9c",
            "exact_attention_blackwell_tma_gb300/csrc/sched.cuh":
                "0328db7053351282b31375c9f4ccf44236a648824c9e57efab5f143fdd22abd6",
            "exact_attention_blackwell_tma_gb300/csrc/kernels.h":
                "5affc1850bc7073eafc4f405d84928b0a015bd41fe555c117e9c97cdf3d90f72",
            "exact_attention_blackwell_tma_gb300/csrc/mask.cuh":
                "a8db3e42b70e326e0df86ce85e11cf81134dc7f609b7d0006d9f1a409692beee",
            "exact_attention_blackwell_tma_gb300/csrc/dq_order.cuh":
                "d3268cfe95ac87277ec035e806c4ac4c57c17361d3c6b4c9c26b3e80fa94ac40",
            "exact_attention_blackwell_tma_gb300/csrc/dq_reduce.cuh":
                "7ddedbe18fcca40f3a3e932502abeb8096da330d02b5731aeb6314e8dafeb072",
        },
    },
    ("b1h32l32768d128", "bwd", True): {
        "bytes": 6605.666e6 + 3768.216e6,
        "profile": "profiles/bwd_kernel_b1h32l32768d128_traffic.md",
        "sources": {
            "exact_attention_blackwell_tma_gb300/csrc/bwd.cu":
                "60bc2511e502cc06be6d193c1279504a2fdce162ce618fc40e08004425c032ba",
            "exact_attention_blackwell_tma_gb300/csrc/ptx.cuh":
                "3c0283284f2342dd722773b9195bbfdc67274aa16994dbb143983c848529bf9c",
            "exact_attention_blackwell_tma_gb300/csrc/sched.cuh":
                "0328db7053351282b31375c9f4ccf44236a648824c9e57efab5f143fdd22abd6",
            "exact_attention_blackwell_tma_gb300/csrc/kernels.h":
                "5affc1850bc7073eafc4f405d84928b0a015bd41fe555c117e9c97cdf3d90f72",
            "exact_attention_blackwell_tma_gb300/csrc/mask.cuh":
                "a8db3e42b70e326e0df86ce85e11cf81134dc7f609b7d0006d9f1a409692beee",
            "exact_attention_blackwell_tma_gb300/csrc/dq_order.cuh":
                "d3268cfe95ac87277ec035e806c4ac4c57c17361d3c6b4c9c26b3e80fa94ac40",
            "exact_attention_blackwell_tma_gb300/csrc/dq_reduce.cuh":
                "7ddedbe18fcca40f3a3e932502abeb8096da330d02b5731aeb6314e8dafeb072",
        },
    },
}


def ncu_traffic(workload, kind, causal):
    """Bytes per launch from NCU_TRAFFIC, or None if absent or the sources changed."""
    import hashlib
    rec = NCU_TRAFFIC.get((workload, kind, causal))
    if rec is None:
        return None
    for rel, digest in rec["sources"].items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    return rec["bytes"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"bf16": float(pk["bf16_tflops"]), "bf16_sustained": float(pk["bf16_tflops_sustained"]),
                "source": "measured"}
    except Exception:
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


class Problem:
    """Device buffers for one workload."""

    def __init__(self, w, device):
        t = inputs.make(w)
        self.w = w
        self.host = t
        self.q, self.k, self.v, self.do = (t[n].to(device) for n in ("q", "k", "v", "do"))
        self.cu = t["cu_seqlens"].to(device) if w.varlen else None
        self.cuk = t["cu_seqlens_k"].to(device) if "cu_seqlens_k" in t else None
        self.mask = inputs.block_mask(w).to(device) if w.block_pattern is not None else None
        self.o = torch.empty(self.q.shape[:-1] + (w.d_v,), dtype=self.q.dtype, device=device)
        self.dq, self.dk, self.dv = torch.empty_like(self.q), torch.empty_like(self.k), torch.empty_like(self.v)
        self.Hkv = w.H_kv
        if w.varlen:
            self.B, self.H, self.Lq, self.Lk, self.d = w.B, w.H, w.total, w.total_k, w.d
            self.lse = torch.empty((w.H, w.total), dtype=torch.float32, device=device)
        else:
            self.B, self.H, self.Lq, self.Lk, self.d = w.B, w.H, w.L, w.L, w.d
            self.lse = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=device)
        ws = max(binding.attn_bwd_ex_workspace_size(self.B, self.H, self.Hkv, self.Lq, self.Lk, self.d, self.w.d_v,
                                                    1, 0), 1)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)

    def clone(self, inputs_from=None):
        """Another buffer set of the same shapes: fresh outputs and workspace;
        fresh inputs, or those of `inputs_from`."""
        c = copy.copy(self)
        for n in ("q", "k", "v", "do"):
            setattr(c, n, getattr(inputs_from, n) if inputs_from is not None else torch.empty_like(getattr(self, n)))
        for n in ("o", "lse", "dq", "dk", "dv", "ws"):
            setattr(c, n, torch.empty_like(getattr(self, n)))
        return c

    def fwd(self, causal):
        if self.cuk is not None:
            rc = binding.attn_fwd_varlen(self.q, self.k, self.v, self.o, self.lse, self.B, self.H, self.Hkv, self.Lq,
                                         self.Lk, self.d, self.w.d_v, self.w.scale, causal, self.cu, self.cuk)
            if rc:
                raise binding.AttnError(rc, binding.last_error())
            return
        rc = binding.attn_fwd_ex(self.q, self.k, self.v, self.o, self.lse, self.B, self.H, self.Hkv, self.Lq,
                                 self.Lk, self.d, self.w.d_v, self.w.scale, causal, self.w.window[0],
                                 self.w.window[1], self.mask, 1, self.cu, None)
        if rc:
            raise binding.AttnError(rc, binding.last_error())

    def bwd(self, causal, deterministic=0):
        if self.cuk is not None:
            rc = binding.attn_bwd_varlen(self.q, self.k, self.v, self.o, self.lse, self.do, self.dq, self.dk,
                                         self.dv, self.B, self.H, self.Hkv, self.Lq, self.Lk, self.d, self.w.scale,
                                         causal, self.cu, self.cuk, deterministic, self.ws, self.ws.numel())
            if rc:
                raise binding.AttnError(rc, binding.last_error())
            return
        rc = binding.attn_bwd_ex(self.q, self.k, self.v, self.o, self.lse, self.do, self.dq, self.dk, self.dv,
                                 self.B, self.H, self.Hkv, self.Lq, self.Lk, self.d, self.w.d_v, self.w.scale, causal,
                                 self.w.window[0], self.w.window[1], self.mask, 1, self.cu, None, deterministic,
                                 self.ws, self.ws.numel())
        if rc:
            raise binding.AttnError(rc, binding.last_error())


class E2EPipeline:
    """Steps through the C ABI from pinned host buffers: every step copies its
    inputs to the device and every mask variant's results back. The copies of
    neighbouring steps overlap the computation: two buffer sets (by step
    parity; outputs also by variant), host-to-device copies on one stream and
    device-to-host copies on another, ordered against the computation by
    events. After run(), outs[parity][variant] hold that step's results."""

    def __init__(self, prob, variants, kinds):
        self.variants, self.kinds = variants, kinds
        ins = ("q", "k", "v", "do") if "bwd" in kinds else ("q", "k", "v")
        self.host = {n: prob.host[n].pin_memory() for n in ins}
        out_names = ("o", "lse", "dq", "dk", "dv") if "bwd" in kinds else ("o", "lse")
        self.base = [prob, prob.clone()]
        self.sets = [[self.base[p] if vi == 0 else self.base[p].clone(inputs_from=self.base[p])
                      for vi in range(len(variants))] for p in range(2)]
        self.outs = [[{n: torch.empty(getattr(s_, n).shape, dtype=getattr(s_, n).dtype, pin_memory=True)
                       for n in out_names} for s_ in row] for row in self.sets]
        self.h2d_bytes = sum(x.numel() * x.element_size() for x in self.host.values())
        self.d2h_bytes = sum(x.numel() * x.element_size() for x in self.outs[0][0].values()) * len(variants)
        self.up, self.down = torch.cuda.Stream(), torch.cuda.Stream()
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.in_free = [torch.cuda.Event() for _ in range(2)]
        self.done = [[torch.cuda.Event() for _ in variants] for _ in range(2)]
        self.out_free = [[torch.cuda.Event() for _ in variants] for _ in range(2)]

    def _upload(self, i):
        p = i % 2
        self.up.wait_event(self.in_free[p])          # the step before that used this set has computed
        with torch.cuda.stream(self.up):
            for n, src in self.host.items():
                getattr(self.base[p], n).copy_(src, non_blocking=True)
        self.in_ready[p].record(self.up)

    def _compute_and_download(self, i):
        p = i % 2
        main = torch.cuda.current_stream()
        main.wait_event(self.in_ready[p])
        for vi, c in enumerate(self.variants):
            s_ = self.sets[p][vi]
            main.wait_event(self.out_free[p][vi])   # this set's previous results are on the host
            for kind in self.kinds:
                s_.fwd(c) if kind == "fwd" else s_.bwd(c)
            self.done[p][vi].record(main)
            self.down.wait_event(self.done[p][vi])
            with torch.cuda.stream(self.down):
                for n, dst in self.outs[p][vi].items():
                    dst.copy_(getattr(s_, n), non_blocking=True)
            self.out_free[p][vi].record(self.down)
        self.in_free[p].record(main)

    def run(self, nsteps, start=None):
        """Enqueue nsteps steps; the current stream then waits for every copy."""
        if start is not None:
            self.up.wait_event(start)
        self._upload(0)
        for i in range(nsteps):
            if i + 1 < nsteps:
                self._upload(i + 1)
            self._compute_and_download(i)
        main = torch.cuda.current_stream()
        for p in range(2):
            for vi in range(len(self.variants)):
                main.wait_event(self.out_free[p][vi])


def flops(w, causal, which):
    ww = w.with_(causal=causal)
    return ww.fwd_flops() if which == "fwd" else ww.bwd_flops()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "power_w_max": max(r[2] for r in rows)}


def dist_setup(backend="nccl"):
    """World size, rank, local rank and the process group module (None for one
    process). Independent replicas: the group only carries the barrier and the
    max over ranks of the timed region, never data."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if backend == "nccl":
        torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend)
        return world, rank, local, dist
    return 1, 0, local, None


def _device_of(dist):
    return "cuda" if dist is None or dist.get_backend() == "nccl" else "cpu"


def max_over_ranks(x, dist):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=_device_of(dist))
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()
    if _device_of(dist) == "cuda":
        torch.cuda.synchronize()


def time_single(prob, call, steps, warmup):
    """Mean CUDA-event time (ms) of one call, on the stream it is launched on,
    over `steps` back-to-back runs after `warmup` untimed ones."""
    return time_single_stats(prob, call, steps, warmup)[0]


def time_single_stats(prob, call, steps, warmup):
    """(mean, median) CUDA-event time (ms) of one call, as time_single."""
    for _ in range(max(warmup, 3)):
        call(prob)
    binding.check_status()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record()
        call(prob)
        b.record()
    torch.cuda.synchronize()
    binding.check_status()
    ts = [a.elapsed_time(b) for a, b in evs]
    return statistics.mean(ts), statistics.median(ts)


def single_call_records(args, pk, dev, main_prob):
    """The goal row (causal forward, d = 128, L = 8192) and the deterministic
    causal backward of the long-context workload, each with its own fraction
    of the measured dense BF16 peak."""
    out = {}
    w, _ = WORKLOADS[TARGET_WORKLOAD]
    prob = main_prob if args.workload == TARGET_WORKLOAD else Problem(w, dev)
    t_ms, t_med = time_single_stats(prob, lambda p_: p_.fwd(True), args.steps, args.warmup)
    fl = flops(w, True, "fwd")
    ach = fl / (t_ms * 1e-3) / 1e12
    out["target"] = {"workload": TARGET_WORKLOAD, "call": "attn_fwd (causal)", "ms": t_ms, "median_ms": t_med,
                     "achieved": ach,
                     "unit": UNIT, "peak": pk["bf16"], "frac": ach / pk["bf16"], "goal_frac": TARGET_FRAC,
                     "met": ach / pk["bf16"] >= TARGET_FRAC,
                     "l2": "inputs 192 MiB > 129 MiB L2; no flush between calls"}
    if prob is not main_prob:
        del prob
        torch.cuda.empty_cache()
    wl, _ = WORKLOADS["b1h32l32768d128"]
    prob = main_prob if args.workload == "b1h32l32768d128" else None
    if prob is not None:
        prob.fwd(True)
        t_ms, t_med = time_single_stats(prob, lambda p_: p_.bwd(True, deterministic=1), args.steps, args.warmup)
        fl = flops(wl, True, "bwd")
        ach = fl / (t_ms * 1e-3) / 1e12
        out["deterministic"] = {"workload": "b1h32l32768d128", "call": "attn_bwd (causal, deterministic)",
                                "ms": t_ms, "median_ms": t_med, "achieved": ach, "unit": UNIT, "peak": pk["bf16"],
                                "frac": ach / pk["bf16"]}
    return out


# ------------------------------------------------------------------------------------------ oracle
# About 10 s of the oracle on 16 host cores (it runs near 0.027 TFLOP/s there).
ORACLE_SAMPLE_FLOPS = 3e11


def oracle_sample(w, variants, nthreads=None, budget=ORACLE_SAMPLE_FLOPS):
    """fp64 oracle (forward + backward) for each variant on the first heads of
    batch entry 0 (varlen: of the longest prefill sequence), as many as the
    sample budget holds; when one whole head would exceed it, on the leading
    L' x L' block of head 0 (the first L' queries and keys; for a causal mask
    exactly the attention of that prefix). Each query head is paired with the
    key/value head it reads. Returns (algorithmic flops of the sample,
    seconds, threads, description)."""
    import numpy as np
    import oracle
    t = inputs.make(w)
    nthreads = nthreads or oracle.default_threads()
    if w.varlen:
        # the longest prefill sequence (queries = keys), head 0
        cu = t["cu_seqlens"]
        cuk = t.get("cu_seqlens_k", cu)
        lq, lk = cu[1:] - cu[:-1], cuk[1:] - cuk[:-1]
        same = [b for b in range(w.B) if int(lq[b]) == int(lk[b])]
        s = max(same, key=lambda b: int(lq[b])) if w.lengths_k is not None else 0
        a, c, L = int(cu[s]), int(cuk[s]), int(lq[s])
        full = {n: t[n][a:a + L].unsqueeze(0) for n in ("q", "do")}
        full.update({n: t[n][c:c + L].unsqueeze(0) for n in ("k", "v")})
        where = f"sequence {s}"
    else:
        L = w.L
        full = {n: t[n][:1] for n in ("q", "k", "v", "do")}
        where = "batch 0"

    def sample_flops(Lp, nh=1):
        sw = w.with_(lengths=None, lengths_k=None, hkv=None, B=1, H=nh, L=Lp)   # (a block pattern scales with L)
        return sum(flops(sw, c, kind) for c in variants for kind in kinds_of(w))

    Lp = L
    while Lp > 128 and sample_flops(Lp) > budget:
        Lp = max(128, (Lp // 2) // 128 * 128)
    nh = max(1, min(w.H, int(budget // sample_flops(Lp)))) if Lp == L else 1
    group = w.H // w.H_kv
    src = {n: full[n][:, :, :nh] for n in ("q", "do")}
    src.update({n: full[n][:, :, [h // group for h in range(nh)]] for n in ("k", "v")})
    where += f", heads 0-{nh - 1}" if nh > 1 else ", head 0"
    f64 = {n: x[:, :Lp].float().numpy().astype(np.float64) for n, x in src.items()}
    total_flops, secs = 0, 0.0
    kinds = kinds_of(w)
    for causal in variants:
        t0 = time.perf_counter()
        bm = None
        if w.block_pattern is not None:   # the leading Lp x Lp block of the mask
            nb = -(-Lp // 128)
            bm = inputs.block_mask(w)[:, :nb, :nb].numpy()
        oracle.fwd(f64["q"], f64["k"], f64["v"], w.scale, causal, nthreads=nthreads, window_left=w.window[0],
                   window_right=w.window[1], block_mask=bm)
        if "bwd" in kinds:
            oracle.bwd(f64["q"], f64["k"], f64["v"], f64["do"], w.scale, causal, nthreads=nthreads,
                       window_left=w.window[0], window_right=w.window[1], block_mask=bm)
        secs += time.perf_counter() - t0
    total_flops = sample_flops(Lp, nh)
    what = f"{where}" + (f", leading {Lp}x{Lp} block" if Lp < L else "") + \
        f" of {w.name}, {'+'.join({'fwd': 'forward', 'bwd': 'backward'}[k] for k in kinds_of(w))}, " + \
        f"{'/'.join('causal' if c else 'non-causal' for c in variants)}"
    return total_flops, secs, nthreads, what


def run_reference(args, world, rank, dist):
    if rank != 0:
        return 0
    w, variants = WORKLOADS[args.workload]
    # the whole run stays near a dozen budgets (about two minutes on 16 cores)
    budget = ORACLE_SAMPLE_FLOPS * min(1.0, 12.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, variants, budget=budget)
    fl, secs = 0, 0.0
    threads, sample = None, ""
    for _ in range(args.steps):
        f, sec, threads, sample = oracle_sample(w, variants, budget=budget)
        fl += f
        secs += sec
    value = fl / secs / 1e12
    sample += ", per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "variants": ["causal" if c else "non-causal" for c in variants]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------ ours
def run_ours(args, world, rank, local, dist):
    w, variants = WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    pk = load_peaks()
    prob = Problem(w, dev)
    kinds = kinds_of(w)
    step_flops = sum(flops(w, c, kind) for c in variants for kind in kinds)
    used = (prob.q, prob.k, prob.v, prob.do) if "bwd" in kinds else (prob.q, prob.k, prob.v)
    input_bytes = sum(x.numel() * x.element_size() for x in used)

    def step(ev=None):
        for c in variants:
            for kind in kinds:
                if ev is not None:
                    ev[(kind, c)][0].record()
                prob.fwd(c) if kind == "fwd" else prob.bwd(c)
                if ev is not None:
                    ev[(kind, c)][1].record()

    for _ in range(max(args.warmup, 3)):
        step()
    binding.check_status()

    # ---- timed region: K steps, per-call events on the launching stream
    evs = [{(k, c): (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for k in kinds for c in variants} for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(dist)
        t0.record()
        for i in range(args.steps):
            step(evs[i])
        t1.record()
        barrier(dist)
    binding.check_status()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, dist)
    value = world * step_flops / (ms * 1e-3) / 1e12

    # per-kernel-call durations -> rooflines
    per_call, per_call_median = {}, {}
    for key in evs[0]:
        ts = [e[key][0].elapsed_time(e[key][1]) for e in evs]
        per_call[key] = statistics.mean(ts)
        per_call_median[key] = statistics.median(ts)
    rooflines = []
    for (kind, c), t_ms in per_call.items():
        fl = flops(w, c, kind)
        ach = fl / (t_ms * 1e-3) / 1e12
        rooflines.append({"kernel": f"attn_{kind}", "variant": "causal" if c else "non-causal",
                          "ms": t_ms, "median_ms": per_call_median[(kind, c)], "achieved": ach,
                          "bound": "tensor", "unit": "TFLOP/s",
                          "peak": pk["bf16"], "frac": ach / pk["bf16"], "traffic": None})
    for r in rooflines:
        r["traffic"] = ncu_traffic(w.name, r["kernel"][5:], r["variant"] == "causal")
    dom = max(rooflines, key=lambda r: r["ms"])
    roofline = {"bound": "tensor", "achieved": dom["achieved"], "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": dom["achieved"] / pk["bf16"], "traffic": dom["traffic"],
                "kernel": f"{dom['kernel']} ({dom['variant']})",
                "peak_source": f"{pk['source']} bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
                "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of the main kernel, per launch"}

    # ---- the goal row and the deterministic backward, one call each
    extra = {} if args.no_extra else single_call_records(args, pk, dev, prob)

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        pipe = E2EPipeline(prob, variants, kinds)
        pipe.run(2)
        barrier(dist)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        pipe.run(args.steps, start=a)
        b.record()
        barrier(dist)
        e_ms = max_over_ranks(a.elapsed_time(b) / args.steps, dist)
        e2e = {"value": world * step_flops / (e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": pipe.h2d_bytes, "d2h_bytes_per_step": pipe.d2h_bytes,
               "overlap": "two buffer sets; host-to-device and device-to-host copies on their own streams"}

    # ---- oracle on the host cores (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, secs, threads, what = oracle_sample(w, variants)
        cpu = {"value": fl / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{what}; {secs:.1f} s", "seconds": secs}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": args.workload, "B": w.B, "H": w.H, "H_kv": w.H_kv, "L": w.L, "d": w.d,
                           "d_v": w.d_v, "window": list(w.window),
                           "calls": list(kinds),
                           "variants": ["causal" if c else "non-causal" for c in variants],
                           "flops_per_step": step_flops,
                           "l2": f"inputs {input_bytes / 2**20:.0f} MiB > 129 MiB L2; no flush between steps",
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
                "frac_of_peak": value / world / pk["bf16"],
                "roofline": roofline, "roofline_calls": rooflines, **extra,
                "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps * len(variants) * (4 if "bwd" in kinds else 1),
                "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the goal-row and deterministic single-call timings")
    args = ap.parse_args()
    world, rank, local, dist = dist_setup() if args.impl == "ours" else (
        int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0, None)
    if args.impl == "reference":
        return run_reference(args, world, rank, dist)
    rc = run_ours(args, world, rank, local, dist)
    if dist is not None:
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
