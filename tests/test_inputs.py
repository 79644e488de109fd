"""The seeded synthetic inputs both the CUDA path and the oracle draw from:
shapes and dtypes for every layout, the same draw for the same seed, the K
spikes the recipe plants, and the length mixes of the packed workloads. No
GPU."""
import torch

from exact_attention_blackwell_tma_gb300 import inputs
from exact_attention_blackwell_tma_gb300.inputs import Workload


def test_dense_shapes_dtypes_and_determinism():
    w = Workload("t", B=2, H=4, L=96, d=64, causal=True, seed=7, dv=128, hkv=2)
    a, b = inputs.make(w), inputs.make(w)
    assert a["q"].shape == (2, 96, 4, 64) and a["k"].shape == (2, 96, 2, 64)
    assert a["v"].shape == (2, 96, 2, 128) and a["do"].shape == (2, 96, 4, 128)
    for n in ("q", "k", "v", "do"):
        assert a[n].dtype == torch.bfloat16
        assert torch.equal(a[n], b[n])
    c = inputs.make(w.with_(seed=8))
    assert not torch.equal(a["q"], c["q"])
    assert "do" not in inputs.make(w, with_grad=False)
    # q, k, v, dO are independent draws
    assert not torch.equal(a["q"][..., :2, :], a["k"])


def test_k_spikes_scale_exactly_the_planted_rows():
    w = Workload("t", B=2, H=2, L=200, d=64, causal=True, seed=3, kspike_frac=0.05, kspike=4.0)
    spiky = inputs.make(w)["k"].float()
    plain = inputs.make(w.with_(kspike_frac=0.0))["k"].float()
    for b in range(2):
        scaled = [i for i in range(200) if not torch.equal(spiky[b, i], plain[b, i])]
        assert len(scaled) == 10                               # round(0.05 * 200) rows per batch entry
        for i in scaled:                                       # x4 is exact in bf16
            assert torch.equal(spiky[b, i], plain[b, i] * 4.0)


def test_varlen_layout_and_offsets():
    lq, lk = (5, 0, 130), (7, 3, 1)
    w = Workload("t", B=3, H=2, L=130, d=64, causal=True, seed=2, lengths=lq, lengths_k=lk, hkv=1)
    t = inputs.make(w)
    assert t["q"].shape == (135, 2, 64) and t["k"].shape == (11, 1, 64) and t["do"].shape == (135, 2, 64)
    assert t["cu_seqlens"].tolist() == [0, 5, 5, 135] and t["cu_seqlens"].dtype == torch.int32
    assert t["cu_seqlens_k"].tolist() == [0, 7, 10, 11]


def test_length_mixes():
    lens = inputs.varlen_lengths(32, 256, 16384, 4)
    assert len(lens) == 32 and all(256 <= L <= 16384 for L in lens)
    assert lens == inputs.varlen_lengths(32, 256, 16384, 4)
    lq, lk = inputs.prefill_decode_lengths(32, 256, 8192, 1024, 16384, 6)
    prefill = [(a, b) for a, b in zip(lq, lk) if a == b]
    decode = [(a, b) for a, b in zip(lq, lk) if a != b]
    assert len(prefill) == 16 and len(decode) == 16
    assert all(256 <= a <= 8192 for a, _ in prefill)
    assert all(1 <= a <= 16 and 1024 <= b <= 16384 for a, b in decode)
    assert inputs.PREFILL_DECODE.lengths == lq and inputs.PREFILL_DECODE.lengths_k == lk


def test_small_problem_shapes():
    t = inputs.small(B=2, H=4, L=33, d=192, Lk=70, dv=128, Hkv=2, seed=9)
    assert t["q"].shape == (2, 33, 4, 192) and t["k"].shape == (2, 70, 2, 192)
    assert t["v"].shape == (2, 70, 2, 128) and t["do"].shape == (2, 33, 4, 128)
