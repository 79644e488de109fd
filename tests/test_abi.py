"""The C ABI library builds, loads without a GPU and exports every declared symbol."""
import ctypes
import os
import re

import pytest

from exact_attention_blackwell_tma_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def built():
    return build.build()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_last_error",
                     "attn_check_status"):
        assert required in names


def test_library_exports_every_declared_symbol(built):
    lib = ctypes.CDLL(binding.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in attn.h but not exported"


def declared_arg_counts():
    """Number of parameters of every function attn.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, args in re.findall(r"\b(attn_\w+)\s*\(([^)]*)\)\s*;", text):
        args = args.strip()
        out[name] = 0 if args in ("", "void") else len(args.split(","))
    return out


def test_binding_declares_the_header_signatures(built):
    """Every ctypes declaration in the binding has the header's argument count."""
    lib = binding.load()
    counts = declared_arg_counts()
    assert len(counts) == len(declared_functions())
    for name, n in counts.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes in the binding"
        assert len(fn.argtypes) == n, f"{name}: binding has {len(fn.argtypes)} arguments, attn.h {n}"


def test_error_codes_match_header(built):
    text = open(HEADER).read()
    codes = dict(re.findall(r"#define (ATTN_\w+) \(?(-?\d+)\)?", text))
    assert int(codes["ATTN_OK"]) == binding.ATTN_OK
    assert int(codes["ATTN_ERR_ARG"]) == binding.ATTN_ERR_ARG
    assert int(codes["ATTN_ERR_ALIGN"]) == binding.ATTN_ERR_ALIGN
    assert int(codes["ATTN_ERR_LAUNCH"]) == binding.ATTN_ERR_LAUNCH
    assert int(codes["ATTN_ERR_WORKSPACE"]) == binding.ATTN_ERR_WORKSPACE
    assert int(codes["ATTN_ERR_TIMEOUT"]) == binding.ATTN_ERR_TIMEOUT


def test_argument_errors_need_no_gpu(built):
    """Host-side validation returns before touching the device."""
    lib = binding.load()
    dummy = 1 << 20   # never dereferenced: validation fails first
    # unsupported head dim
    assert lib.attn_fwd(dummy, dummy, dummy, dummy, dummy, 1, 1, 128, 128, 96, 0.1, 0, None, None) == -1
    assert "head dim" in binding.last_error()
    # non-positive scale
    assert lib.attn_fwd(dummy, dummy, dummy, dummy, dummy, 1, 1, 128, 128, 64, 0.0, 0, None, None) == -1
    # null pointer
    assert lib.attn_fwd(None, dummy, dummy, dummy, dummy, 1, 1, 128, 128, 64, 0.1, 0, None, None) == -1
    # misaligned pointer
    assert lib.attn_fwd(dummy + 2, dummy, dummy, dummy, dummy, 1, 1, 128, 128, 64, 0.1, 0, None, None) == -2
    # varlen requires Lq == Lk (both the packed row count)
    assert lib.attn_fwd(dummy, dummy, dummy, dummy, dummy, 2, 1, 128, 64, 64, 0.1, 0, dummy, None) == -1
    # varlen batches: 1 .. 1024 sequences (the sequence map's capacity)
    assert lib.attn_fwd(dummy, dummy, dummy, dummy, dummy, 1025, 1, 4096, 4096, 64, 0.1, 0, dummy, None) == -1
    assert "1024" in binding.last_error()
    assert lib.attn_fwd(dummy, dummy, dummy, dummy, dummy, 0, 1, 4096, 4096, 64, 0.1, 0, dummy, None) == -1
    assert lib.attn_fwd_varlen(dummy, dummy, dummy, dummy, dummy, 1025, 1, 1, 4096, 4096, 64, 64, 0.1, 0, dummy,
                               dummy, None) == -1
    # separate value head dim: only (192, 128) besides dv = d
    assert lib.attn_fwd_hdim(dummy, dummy, dummy, dummy, dummy, 1, 1, 128, 128, 128, 64, 0.1, 0, None, None) == -1
    assert "dv=64" in binding.last_error()
    assert lib.attn_fwd_hdim(dummy + 2, dummy, dummy, dummy, dummy, 1, 1, 128, 128, 192, 128, 0.1, 0, None,
                             None) == -2
    # grouped heads: the key/value heads must divide the query heads
    assert lib.attn_fwd_gqa(dummy, dummy, dummy, dummy, dummy, 1, 6, 4, 128, 128, 128, 128, 0.1, 0, None,
                            None) == -1
    assert "key/value heads 4" in binding.last_error()
    assert lib.attn_fwd_gqa(dummy, dummy, dummy, dummy, dummy, 1, 4, 0, 128, 128, 128, 128, 0.1, 0, None,
                            None) == -1
    assert lib.attn_fwd_gqa(dummy, dummy, dummy, dummy, dummy, 1, 2, 4, 128, 128, 128, 128, 0.1, 0, None,
                            None) == -1
    assert lib.attn_bwd_gqa(*([dummy] * 9), 1, 8, 3, 128, 128, 64, 0.1, 0, None, 0, dummy, 1 << 30, None) == -1
    # block masks: dense problems only, one mask or one per query head
    assert lib.attn_fwd_ex(dummy, dummy, dummy, dummy, dummy, 2, 4, 4, 256, 256, 64, 64, 0.1, 1, -1, -1, dummy, 1,
                           dummy, None, None) == -1
    assert "dense" in binding.last_error()
    assert lib.attn_fwd_ex(dummy, dummy, dummy, dummy, dummy, 1, 4, 4, 256, 256, 64, 64, 0.1, 1, -1, -1, dummy, 3,
                           None, None, None) == -1
    assert lib.attn_fwd_ex(dummy, dummy, dummy, dummy, dummy, 1, 4, 4, 256, 256, 64, 64, 0.1, 1, -2, -1, None, 1,
                           None, None, None) == -1
    # backward: workspace too small
    ws = lib.attn_bwd_workspace_size(1, 1, 128, 128, 64, 0, 0)
    assert ws > 0
    rc = lib.attn_bwd(*([dummy] * 9), 1, 1, 128, 128, 64, 0.1, 0, None, 0, dummy, ws - 1, None)
    assert rc == -4


def test_workspace_size_grows_with_problem(built):
    lib = binding.load()
    a = lib.attn_bwd_workspace_size(1, 16, 4096, 4096, 128, 1, 0)
    b = lib.attn_bwd_workspace_size(4, 16, 4096, 4096, 128, 1, 0)
    assert b > a > 4 * 16 * 4096 * 128 // 4   # at least the fp32 dQ accumulator
    assert lib.attn_bwd_workspace_size(-1, 1, 1, 1, 64, 0, 0) == 0
    # grouped heads: Hkv = H is the plain size; few key/value heads add partial dK/dV slots
    mha = lib.attn_bwd_workspace_size(2, 16, 8192, 8192, 128, 1, 0)
    assert lib.attn_bwd_gqa_workspace_size(2, 16, 16, 8192, 8192, 128, 1, 0) == mha
    assert lib.attn_bwd_gqa_workspace_size(2, 16, 2, 8192, 8192, 128, 1, 0) > mha
    assert lib.attn_bwd_gqa_workspace_size(2, 16, 3, 8192, 8192, 128, 1, 0) == 0


@pytest.mark.parametrize("B,H,Hkv,L,d,split", [
    (2, 16, 2, 8192, 128, 4),    # 256 key-block tiles: 4 tiles per key block reach 640
    (2, 16, 1, 8192, 128, 8),    # multi-query: 128 tiles, split 8
    (5, 32, 16, 1024, 64, 1),    # 640 tiles already
    (2, 4, 2, 300, 64, 2),       # small: the whole group is split
    (1, 6, 2, 256, 128, 3),      # the group size when no divisor reaches the target
])
def test_grouped_split_policy(built, B, H, Hkv, L, d, split):
    """The partial dK/dV slots in the workspace follow the split rule of the
    header: the smallest divisor of H / Hkv giving at least 640 work tiles."""
    lib = binding.load()
    base = lib.attn_bwd_gqa_workspace_size(B, H, H, L, L, d, 1, 0)
    got = lib.attn_bwd_gqa_workspace_size(B, H, Hkv, L, L, d, 1, 0)
    part = 2 * split * B * L * Hkv * d * 4 if split > 1 else 0
    assert got - base == (part + 255) // 256 * 256


@pytest.mark.parametrize("B,H,T,d,dv", [(3, 4, 1000, 64, 64), (32, 16, 200000, 128, 128), (7, 2, 129, 192, 128),
                                        (1, 1, 1, 256, 256)])
def test_workspace_holds_every_part(built, B, H, T, d, dv):
    """A lower bound built from the parts the backward keeps in the workspace,
    for a packed batch of T rows (the largest layout): the fp32 dQ
    accumulator, D, two semaphores per dQ tile of each sequence (a sequence's
    ragged last block included: H * (T / 128 + B + 1) tiles), and the sequence
    map (four arrays of about 1024 ints)."""
    lib = binding.load()
    got = lib.attn_bwd_ex_workspace_size(B, H, H, T, T, d, dv, 1, 1)
    need = 4 * T * H * d + 4 * T * H + 4 * 2 * H * (T // 128 + B + 1) + 4 * 4 * 1024
    assert got >= need
    assert got % 256 == 0


def test_exp2_emulation_setting(built):
    """attn_set_exp2_emulation: head dims 64 and 128, one pair in 0, 4 or 8;
    returns the previous setting; anything else is an argument error."""
    lib = binding.load()
    prev = lib.attn_set_exp2_emulation(128, 8)
    assert prev in (0, 4, 8)
    assert lib.attn_set_exp2_emulation(128, 4) == 8
    assert lib.attn_set_exp2_emulation(128, prev) == 4
    assert lib.attn_set_exp2_emulation(192, 8) == binding.ATTN_ERR_ARG
    assert lib.attn_set_exp2_emulation(64, 3) == binding.ATTN_ERR_ARG
    assert "0 (off), 4 or 8" in binding.last_error()
