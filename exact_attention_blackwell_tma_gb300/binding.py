"""Python binding of libattn.so: the C entry points under the same names.

Argument marshalling only: every step of the computation runs in the CUDA
library. PyTorch supplies device memory and the current stream. If the
library has not been built, ``load()`` raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None
_selftest = None

c_int, c_float, c_size_t, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

ATTN_OK, ATTN_ERR_ARG, ATTN_ERR_ALIGN, ATTN_ERR_LAUNCH, ATTN_ERR_WORKSPACE, ATTN_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"attn error {code}: {msg}")
        self.code = code


def _declare(lib):
    lib.attn_fwd.restype = c_int
    lib.attn_fwd.argtypes = [c_void_p] * 5 + [c_int] * 5 + [c_float, c_int, c_void_p, c_void_p]
    lib.attn_fwd_hdim.restype = c_int
    lib.attn_fwd_hdim.argtypes = [c_void_p] * 5 + [c_int] * 6 + [c_float, c_int, c_void_p, c_void_p]
    lib.attn_fwd_gqa.restype = c_int
    lib.attn_fwd_gqa.argtypes = [c_void_p] * 5 + [c_int] * 7 + [c_float, c_int, c_void_p, c_void_p]
    lib.attn_fwd_ex.restype = c_int
    lib.attn_fwd_ex.argtypes = ([c_void_p] * 5 + [c_int] * 7 + [c_float, c_int, c_int, c_int, c_void_p, c_int,
                                                                  c_void_p, c_void_p, c_void_p])
    lib.attn_bwd_ex_workspace_size.restype = c_size_t
    lib.attn_bwd_ex_workspace_size.argtypes = [c_int] * 9
    lib.attn_bwd_ex.restype = c_int
    lib.attn_bwd_ex.argtypes = ([c_void_p] * 9 + [c_int] * 7 + [c_float, c_int, c_int, c_int, c_void_p, c_int,
                                                                  c_void_p, c_void_p, c_int, c_void_p, c_size_t,
                                                                  c_void_p])
    lib.attn_fwd_varlen.restype = c_int
    lib.attn_fwd_varlen.argtypes = [c_void_p] * 5 + [c_int] * 7 + [c_float, c_int, c_void_p, c_void_p, c_void_p]
    lib.attn_bwd_workspace_size.restype = c_size_t
    lib.attn_bwd_workspace_size.argtypes = [c_int] * 7
    lib.attn_bwd.restype = c_int
    lib.attn_bwd.argtypes = ([c_void_p] * 9 + [c_int] * 5 + [c_float, c_int, c_void_p, c_int, c_void_p, c_size_t,
                                                               c_void_p])
    lib.attn_bwd_gqa_workspace_size.restype = c_size_t
    lib.attn_bwd_gqa_workspace_size.argtypes = [c_int] * 8
    lib.attn_bwd_gqa.restype = c_int
    lib.attn_bwd_gqa.argtypes = ([c_void_p] * 9 + [c_int] * 6 + [c_float, c_int, c_void_p, c_int, c_void_p,
                                                                   c_size_t, c_void_p])
    lib.attn_bwd_varlen.restype = c_int
    lib.attn_bwd_varlen.argtypes = ([c_void_p] * 9 + [c_int] * 6 + [c_float, c_int, c_void_p, c_void_p, c_int,
                                                                      c_void_p, c_size_t, c_void_p])
    lib.attn_bwd_noalloc.restype = c_int
    lib.attn_bwd_noalloc.argtypes = [c_void_p] * 9 + [c_int] * 5 + [c_float, c_int, c_void_p, c_int, c_void_p]
    lib.attn_set_backward_cta_pairs.restype = c_int
    lib.attn_set_backward_cta_pairs.argtypes = [c_int]
    lib.attn_set_exp2_emulation.restype = c_int
    lib.attn_set_exp2_emulation.argtypes = [c_int, c_int]
    lib.attn_last_error.restype = ctypes.c_char_p
    lib.attn_last_error.argtypes = []
    lib.attn_check_status.restype = c_int
    lib.attn_check_status.argtypes = [c_void_p]
    lib.attn_version.restype = c_int
    lib.attn_version.argtypes = []
    return lib


def library_path() -> str:
    return _build.lib_path("libattn.so")


def load():
    """Load libattn.so (built by ``build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: run exact_attention_blackwell_tma_gb300.build.build() "
                                   "(or __graft_entry__.build()) first; there is no CPU fallback")
            _lib = _declare(ctypes.CDLL(path))
    return _lib


def load_selftest():
    global _selftest
    with _lock:
        if _selftest is None:
            path = _build.lib_path("libattn_selftest.so")
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build first")
            lib = ctypes.CDLL(path)
            lib.attn_selftest_mma.restype = c_int
            lib.attn_selftest_mma.argtypes = [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
            lib.attn_selftest_exp2.restype = c_int
            lib.attn_selftest_exp2.argtypes = [c_void_p, c_void_p, c_void_p, c_int, c_void_p]
            lib.attn_selftest_wait_timeout.restype = c_int
            lib.attn_selftest_wait_timeout.argtypes = [c_void_p, ctypes.c_ulonglong, c_void_p]
            _selftest = lib
    return _selftest


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def last_error() -> str:
    return load().attn_last_error().decode()


def _check(rc: int):
    if rc != ATTN_OK:
        raise AttnError(rc, last_error())


# ---------------------------------------------------------------- C entry points, same names

def attn_fwd(q, k, v, o, lse, B, H, Lq, Lk, d, scale, causal, cu_seqlens=None, stream=None) -> int:
    return load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Lq, Lk, d, scale, int(causal),
                           _ptr(cu_seqlens), _stream(stream))

def attn_fwd_hdim(q, k, v, o, lse, B, H, Lq, Lk, d, dv, scale, causal, cu_seqlens=None, stream=None) -> int:
    return load().attn_fwd_hdim(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Lq, Lk, d, dv, scale,
                                int(causal), _ptr(cu_seqlens), _stream(stream))


def attn_fwd_gqa(q, k, v, o, lse, B, H, Hkv, Lq, Lk, d, dv, scale, causal, cu_seqlens=None, stream=None) -> int:
    return load().attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Lq, Lk, d, dv, scale,
                               int(causal), _ptr(cu_seqlens), _stream(stream))


def attn_fwd_varlen(q, k, v, o, lse, B, H, Hkv, Tq, Tk, d, dv, scale, causal, cu_seqlens_q, cu_seqlens_k,
                    stream=None) -> int:
    return load().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Tq, Tk, d, dv, scale,
                                  int(causal), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _stream(stream))


def attn_fwd_ex(q, k, v, o, lse, B, H, Hkv, Lq, Lk, d, d_v, scale, causal, window_left=-1, window_right=-1,
                block_mask=None, mask_heads=1, cu_seqlens_q=None, cu_seqlens_k=None, stream=None) -> int:
    return load().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Lq, Lk, d, d_v, scale,
                              int(causal), int(window_left), int(window_right), _ptr(block_mask), int(mask_heads),
                              _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _stream(stream))


def attn_bwd_ex_workspace_size(B, H, Hkv, Lq, Lk, d, d_v, causal, deterministic) -> int:
    return load().attn_bwd_ex_workspace_size(B, H, Hkv, Lq, Lk, d, d_v, int(causal), int(deterministic))


def attn_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Lq, Lk, d, d_v, scale, causal, window_left,
                window_right, block_mask, mask_heads, cu_seqlens_q, cu_seqlens_k, deterministic, workspace, ws_bytes,
                stream=None) -> int:
    return load().attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                              _ptr(dv), B, H, Hkv, Lq, Lk, d, d_v, scale, int(causal), int(window_left),
                              int(window_right), _ptr(block_mask), int(mask_heads), _ptr(cu_seqlens_q),
                              _ptr(cu_seqlens_k), int(deterministic), _ptr(workspace), ws_bytes, _stream(stream))


def attn_bwd_workspace_size(B, H, Lq, Lk, d, causal, deterministic) -> int:
    return load().attn_bwd_workspace_size(B, H, Lq, Lk, d, int(causal), int(deterministic))


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Lq, Lk, d, scale, causal, cu_seqlens, deterministic,
             workspace, ws_bytes, stream=None) -> int:
    return load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                           _ptr(dv), B, H, Lq, Lk, d, scale, int(causal), _ptr(cu_seqlens), int(deterministic),
                           _ptr(workspace), ws_bytes, _stream(stream))


def attn_bwd_gqa_workspace_size(B, H, Hkv, Lq, Lk, d, causal, deterministic) -> int:
    return load().attn_bwd_gqa_workspace_size(B, H, Hkv, Lq, Lk, d, int(causal), int(deterministic))


def attn_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Lq, Lk, d, scale, causal, cu_seqlens, deterministic,
                 workspace, ws_bytes, stream=None) -> int:
    return load().attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                               _ptr(dv), B, H, Hkv, Lq, Lk, d, scale, int(causal), _ptr(cu_seqlens),
                               int(deterministic), _ptr(workspace), ws_bytes, _stream(stream))


def attn_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Tq, Tk, d, scale, causal, cu_seqlens_q,
                    cu_seqlens_k, deterministic, workspace, ws_bytes, stream=None) -> int:
    return load().attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                  _ptr(dv), B, H, Hkv, Tq, Tk, d, scale, int(causal), _ptr(cu_seqlens_q),
                                  _ptr(cu_seqlens_k), int(deterministic), _ptr(workspace), ws_bytes,
                                  _stream(stream))


def attn_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H, Lq, Lk, d, scale, causal, cu_seqlens,
                     deterministic, stream=None) -> int:
    """attn_bwd without a workspace: scratch comes from a fixed array inside the
    library (for callers that cannot allocate device memory; see include/attn.h)."""
    return load().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                   _ptr(dk), _ptr(dv), B, H, Lq, Lk, d, scale, int(causal), _ptr(cu_seqlens),
                                   int(deterministic), _stream(stream))


def attn_set_backward_cta_pairs(enable) -> int:
    """Backward main kernel on CTA pairs (2-CTA tensor cores) where it applies;
    returns the previous setting."""
    return load().attn_set_backward_cta_pairs(int(bool(enable)))


def attn_set_exp2_emulation(d, every) -> int:
    """Forward exp2 emulation for head dim d: one column pair in `every` (0, 4, 8)
    by the FMA polynomial; returns the previous setting (or a negative code)."""
    return load().attn_set_exp2_emulation(int(d), int(every))


def attn_last_error() -> str:
    return last_error()


def attn_check_status(stream=None) -> int:
    return load().attn_check_status(_stream(stream))


# ---------------------------------------------------------------- tensor-level helpers

def _dims(q, k, cu_seqlens):
    """B, H, Lq, Lk, d and the key/value heads Hkv."""
    if cu_seqlens is None:
        B, Lq, H, d = q.shape
        return B, H, Lq, k.shape[1], d, k.shape[2]
    T, H, d = q.shape
    return cu_seqlens.numel() - 1, H, T, k.shape[0], d, k.shape[1]


def _mask_heads(block_mask, H, Lq, Lk):
    """Heads of a block mask after checking its shape [Hm, ceil(Lq/128), ceil(Lk/128)] (2-D: Hm = 1)."""
    if block_mask is None:
        return 1
    shape = tuple(block_mask.shape)
    want = (-(-Lq // 128), -(-Lk // 128))
    if block_mask.dtype != torch.uint8 or not (shape == want or (len(shape) == 3 and shape[1:] == want
                                                                 and shape[0] in (1, H))):
        raise ValueError(f"block_mask must be uint8 [1 or {H}, {want[0]}, {want[1]}], got {block_mask.dtype} {shape}")
    return 1 if len(shape) == 2 else shape[0]


def _check_tensors(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")


def forward(q, k, v, causal: bool, scale: float | None = None, cu_seqlens=None, out=None, lse=None,
            stream=None, cu_seqlens_k=None, window=(-1, -1), block_mask=None):
    """O, LSE for bf16 q, k, v ([B, L, H, d], or [T, H, d] with int32 cu_seqlens).
    v (and O) may have a head dim of their own (d = 192 with 128); k and v may
    have fewer heads than q (grouped heads: query head h reads h // (H // Hkv)).
    cu_seqlens_k: key offsets of a varlen batch whose key lengths differ.
    window: (left, right) bounds of a local window, -1 for an open side.
    block_mask: uint8 CUDA tensor [Hm, ceil(Lq/128), ceil(Lk/128)] (Hm 1 or H;
    2-D means Hm = 1), dense problems only; zero drops a 128 x 128 block."""
    _check_tensors(q, k, v, cu_seqlens, cu_seqlens_k)
    B, H, Lq, Lk, d, Hkv = _dims(q, k, cu_seqlens)
    dv = v.shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        out = torch.empty(q.shape[:-1] + (dv,), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Lq) if cu_seqlens is None else (H, Lq), dtype=torch.float32, device=q.device)
    if tuple(window) != (-1, -1) or block_mask is not None:
        mh = _mask_heads(block_mask, H, Lq, Lk)
        _check_tensors(block_mask)
        _check(attn_fwd_ex(q, k, v, out, lse, B, H, Hkv, Lq, Lk, d, dv, scale, causal, window[0], window[1],
                           block_mask, mh, cu_seqlens, cu_seqlens_k, stream))
    elif cu_seqlens_k is not None:
        _check(attn_fwd_varlen(q, k, v, out, lse, B, H, Hkv, Lq, Lk, d, dv, scale, causal, cu_seqlens,
                               cu_seqlens_k, stream))
    elif Hkv != H:
        _check(attn_fwd_gqa(q, k, v, out, lse, B, H, Hkv, Lq, Lk, d, dv, scale, causal, cu_seqlens, stream))
    elif dv == d:
        _check(attn_fwd(q, k, v, out, lse, B, H, Lq, Lk, d, scale, causal, cu_seqlens, stream))
    else:
        _check(attn_fwd_hdim(q, k, v, out, lse, B, H, Lq, Lk, d, dv, scale, causal, cu_seqlens, stream))
    return out, lse


def backward(q, k, v, o, lse, dout, causal: bool, scale: float | None = None, cu_seqlens=None,
             deterministic: bool = False, workspace=None, dq=None, dk=None, dv=None, stream=None,
             cu_seqlens_k=None, window=(-1, -1), block_mask=None):
    """dQ, dK, dV (bf16) for the loss sum(O * dO); k and v may have fewer heads
    than q (grouped heads), dK and dV then have theirs; v (dO, dV) may have a head
    dim of its own (d = 192 with 128). cu_seqlens_k, window and block_mask as in forward()."""
    _check_tensors(q, k, v, o, lse, dout, cu_seqlens, cu_seqlens_k)
    B, H, Lq, Lk, d, Hkv = _dims(q, k, cu_seqlens)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    d_v = v.shape[-1]
    need = attn_bwd_ex_workspace_size(B, H, Hkv, Lq, Lk, d, d_v, causal, deterministic)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = workspace.numel() * workspace.element_size()
    if d_v != d or tuple(window) != (-1, -1) or block_mask is not None:
        mh = _mask_heads(block_mask, H, Lq, Lk)
        _check_tensors(block_mask)
        _check(attn_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Lq, Lk, d, d_v, scale, causal, window[0],
                           window[1], block_mask, mh, cu_seqlens, cu_seqlens_k, deterministic, workspace, ws_bytes,
                           stream))
    elif cu_seqlens_k is not None:
        _check(attn_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Lq, Lk, d, scale, causal, cu_seqlens,
                               cu_seqlens_k, deterministic, workspace, ws_bytes, stream))
    elif Hkv != H:
        _check(attn_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Lq, Lk, d, scale, causal, cu_seqlens,
                            deterministic, workspace, ws_bytes, stream))
    else:
        _check(attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Lq, Lk, d, scale, causal, cu_seqlens,
                        deterministic, workspace, ws_bytes, stream))
    return dq, dk, dv


def check_status(stream=None):
    _check(attn_check_status(stream))
