"""The benchmark's end-to-end pipeline (host copies overlapped with the
neighbouring steps' computation on two streams) returns, for every step and
mask variant, exactly the results of the same calls made one after another
on the device: no copy races its computation."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_attention_blackwell_tma_gb300 import inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("steps", [1, 2, 5])
def test_pipelined_steps_return_the_device_results(steps):
    w = inputs.MHA4K.with_(B=1, H=4, L=1024)
    variants, kinds = (True, False), ("fwd", "bwd")
    prob = bench.Problem(w, torch.device("cuda"))
    pipe = bench.E2EPipeline(prob, variants, kinds)
    pipe.run(steps)
    torch.cuda.synchronize()
    ref = bench.Problem(w, torch.device("cuda"))
    last = (steps - 1) % 2
    for vi, c in enumerate(variants):
        ref.fwd(c)
        ref.bwd(c)
        torch.cuda.synchronize()
        for n, got in pipe.outs[last][vi].items():
            assert torch.equal(got, getattr(ref, n).cpu()) or n == "dq", (steps, c, n)
        # dQ accumulates with atomics: compare it within its rounding instead of bit for bit
        dq = pipe.outs[last][vi]["dq"].float()
        assert torch.allclose(dq, ref.dq.cpu().float(), atol=2e-2, rtol=2e-2), (steps, c, "dq")
