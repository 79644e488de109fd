"""GPU self-tests of the device primitives (separate test library)."""
import numpy as np
import pytest
import torch

from exact_attention_blackwell_tma_gb300 import binding

pytestmark = pytest.mark.gpu


def _mma_expected(mode, A, B):
    a, b = A.double(), B.double()
    if mode in (0, 4):
        return a @ b.T
    if mode in (1, 2):
        return a @ b
    return a.T @ b   # mode 3


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_tcgen05_operand_layouts(mode):
    st = binding.load_selftest()
    g = torch.Generator("cpu").manual_seed(100 + mode)
    A = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    B = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    dA, dB = A.cuda(), B.cuda()
    C = torch.full((128, 128), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = st.attn_selftest_mma(mode, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), status.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = _mma_expected(mode, A, B).numpy()
    got = C.double().cpu().numpy()
    err = np.abs(got - ref).max()
    assert err < 1e-3 * np.abs(ref).max() + 1e-3, f"mode {mode}: max err {err}"


def test_bounded_wait_gives_up_and_context_survives():
    st = binding.load_selftest()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = st.attn_selftest_wait_timeout(status.data_ptr(), 20_000_000,   # 20 ms
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 1   # timeout recorded, kernel returned
    # the context is still usable: a normal call runs and the status word is clean
    q = torch.randn(1, 128, 1, 64, device="cuda").to(torch.bfloat16)
    o, lse = binding.forward(q, q, q, causal=False)
    binding.check_status()
    assert torch.isfinite(o.float()).all()
