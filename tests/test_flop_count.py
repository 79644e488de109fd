"""The FLOP count every reported TFLOP/s figure divides by: the number of
unmasked (query, key) pairs of a workload, against closed forms and a
brute-force scan of the mask definition (causal bottom-right aligned, local
windows, block masks, packed sequences with key lengths of their own), and
the per-pair FLOPs of the forward (S and P V) and the backward (five
products). No GPU."""
import pytest

from exact_attention_blackwell_tma_gb300 import inputs
from exact_attention_blackwell_tma_gb300.inputs import Workload


def brute_pairs(lq, lk, causal, wl, wr, mask=None):
    if causal:
        wr = 0
    n = 0
    for i in range(lq):
        for j in range(lk):
            if wr >= 0 and j > i + (lk - lq) + wr:
                continue
            if wl >= 0 and j < i + (lk - lq) - wl:
                continue
            if mask is not None and not mask[i // 128][j // 128]:
                continue
            n += 1
    return n


def test_closed_forms():
    w = Workload("t", B=2, H=3, L=300, d=64, causal=False, seed=0)
    assert w.pairs() == 2 * 3 * 300 * 300
    assert w.with_(causal=True).pairs() == 2 * 3 * 300 * 301 // 2
    assert w.fwd_flops() == 4 * 64 * w.pairs()
    assert w.bwd_flops() == 10 * 64 * w.pairs()        # 2.5x the forward


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [(-1, -1), (0, 0), (50, 0), (-1, 70), (100, 20), (400, -1)])
def test_windows_against_brute_force(causal, window):
    w = Workload("t", B=1, H=2, L=300, d=64, causal=causal, seed=0, window=window)
    assert w.pairs() == 2 * brute_pairs(300, 300, causal, *window)


@pytest.mark.parametrize("causal,window", [(True, (-1, -1)), (False, (-1, -1)), (True, (200, -1)), (False, (90, 90))])
def test_block_mask_against_brute_force(causal, window):
    w = Workload("t", B=2, H=1, L=600, d=64, causal=causal, seed=0, window=window,
                 block_pattern=("local_strided", 2, 3))
    mask = inputs.block_mask(w)[0].tolist()
    assert len(mask) == 5 and len(mask[0]) == 5
    assert w.pairs() == 2 * brute_pairs(600, 600, causal, *window, mask=mask)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_sequences_with_key_lengths_of_their_own(causal):
    lq, lk = (1, 130, 300, 0, 77), (300, 1, 130, 5, 77)
    w = Workload("t", B=len(lq), H=3, L=300, d=128, causal=causal, seed=0, lengths=lq, lengths_k=lk)
    assert w.pairs() == 3 * sum(brute_pairs(a, b, causal, -1, -1) for a, b in zip(lq, lk))


def test_value_head_dim_of_its_own():
    w = Workload("t", B=1, H=2, L=256, d=192, causal=True, seed=0, dv=128)
    p = w.pairs()
    assert w.fwd_flops() == 2 * (192 + 128) * p
    assert w.bwd_flops() == 2 * (3 * 192 + 2 * 128) * p
