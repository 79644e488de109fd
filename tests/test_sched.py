"""Host-side checks of the persistent tile scheduler.

tests/sched_host.cu includes the scheduler's index functions (csrc/sched.cuh,
compiled for the host) and checks, without a GPU: every tile index goes to
exactly one CTA in increasing order (boustrophedon hand-out); the dense
walks (L2-section order, longest-first order) enumerate every (batch, head,
row block) exactly once; the varlen walk covers every tile of a longest-first
sequence map; and the per-CTA work of the benchmark's causal workloads stays
within 3% of the mean. It also checks the mask band's index arithmetic
(csrc/mask.cuh: the keys a row sees, the rows a key is seen by, and the
blocks a group of rows or keys reaches) against a scan of the mask for no
mask, causal and local windows, square and rectangular; and the
deterministic backward's dQ order (csrc/dq_order.cuh): for every dQ tile the
key blocks that contribute to it, found by scanning the mask (and a block
mask), get the turns 0 .. K-1 once each, and every dQ tile's semaphore (both
column chunks in the wide kernel) is its own and lies inside the array the
host sizes, for dense and packed layouts.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "exact_attention_blackwell_tma_gb300", "csrc")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    pytest.skip("nvcc not found")


def test_scheduler_coverage_order_and_balance(tmp_path):
    exe = tmp_path / "sched_host"
    build = subprocess.run([_nvcc(), "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "sched_host.cu"),
                            "-o", str(exe)], capture_output=True, text=True)
    assert build.returncode == 0, build.stdout + build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip().endswith("OK"), run.stdout + run.stderr
