"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never imports, links or
calls it, and this package imports nothing from the CUDA library.

It wraps ``oracle.c`` (plain C loops in double precision, the textbook
definition of O, LSE, dQ, dK, dV; see that file's header for the formulas and
their sources in the FlashAttention-4 paper). The shared object is compiled
with gcc on first use (or by ``build()``) next to the source.

Arrays are numpy, any real dtype (converted to float64; bf16 values widen
exactly). Layouts: dense q/o/dq ``[B, Lq, H, d]``, k/v/dk/dv ``[B, Lk, Hkv, d]``,
lse ``[B, H, Lq]``; varlen (``cu_seqlens`` given for the queries, and
``cu_seqlens_k`` for the keys when their lengths differ) q ``[Tq, H, d]``,
k ``[Tk, Hkv, d]`` and lse ``[H, Tq]``.

Every function here has pins in ``tests/test_oracle_pins.py`` (closed forms,
a textbook softmax restatement, finite differences, invariants); none is
parity-unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)
_bp = ctypes.POINTER(ctypes.c_ubyte)


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared object (gcc, -O2, plain C11)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                           "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Load a compiled oracle shared object and declare its C signatures."""
    lib = ctypes.CDLL(path)
    lib.oracle_fwd.restype = ctypes.c_int
    lib.oracle_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp,
                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, _bp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               _ip, _ip, _ip, ctypes.c_int, ctypes.c_int]
    lib.oracle_bwd.restype = ctypes.c_int
    lib.oracle_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp,
                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, _bp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               _ip, _ip, _ip, ctypes.c_int, _ip, ctypes.c_int, ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


_EMPTY_I32 = np.zeros(1, dtype=np.int32)


def _ptr(a, typ):
    if a is None:
        return None
    if a.size == 0:  # an empty subset must still be a non-NULL pointer
        a = _EMPTY_I32
    return a.ctypes.data_as(typ)


def _dims(q, k, cu, cuk=None):
    """B, H (query heads), Hkv (key/value heads), Lq, Lk, d."""
    if cu is None:
        if q.ndim != 4 or k.ndim != 4:
            raise ValueError("dense tensors must be [B, L, H, d]")
        B, Lq, H, d = q.shape
        Lk, Hkv = k.shape[1], k.shape[2]
        if k.shape[0] != B or k.shape[3] != d:
            raise ValueError("q/k shape mismatch")
    else:
        if q.ndim != 3:
            raise ValueError("varlen tensors must be [T, H, d]")
        T, H, d = q.shape
        Hkv = k.shape[1]
        B = len(cu) - 1
        ck = cu if cuk is None else cuk
        if len(ck) != len(cu):
            raise ValueError("cu_seqlens_k must have the length of cu_seqlens")
        if cu[-1] != T or k.shape[0] != ck[-1] or k.shape[2] != d:
            raise ValueError("cu_seqlens[-1] (cu_seqlens_k[-1]) must equal the packed query (key) length")
        Lq = int(np.max(np.diff(cu))) if B > 0 else 0
        Lk = int(np.max(np.diff(ck))) if B > 0 else 0
    if Hkv < 1 or H % Hkv != 0:
        raise ValueError("query heads must be a multiple of key/value heads")
    return B, H, Hkv, Lq, Lk, d

def _block_mask(mask, H, Lq, Lk, block):
    """(pointer, heads, block_q, block_k) of an optional block mask [Hm, nqb, nkb]."""
    if mask is None:
        return None, 1, 1, 1
    bq, bk = block
    m = np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
    if m.ndim == 2:
        m = m[None]
    if m.shape[0] not in (1, H) or m.shape[1:] != ((Lq + bq - 1) // bq, (Lk + bk - 1) // bk):
        raise ValueError(f"block mask of shape {m.shape} does not match H={H}, Lq={Lq}, Lk={Lk}, block={block}")
    return m, m.shape[0], bq, bk


def _dv(v, k):
    """Head dim of v (may differ from that of q and k); v must match k otherwise."""
    if v.shape[:-1] != k.shape[:-1]:
        raise ValueError("v must have the rows and heads of k")
    return v.shape[-1]


def fwd(q, k, v, scale: float, causal: bool, cu_seqlens=None, rows=None, nthreads=None, cu_seqlens_k=None,
        window_left: int = -1, window_right: int = -1, block_mask=None, block=(128, 128)):
    """O and LSE (natural log) by the definition. Returns (o, lse) as float64.

    q and k share a head dim; v (and O) may have another one; k and v may have
    fewer heads (grouped heads). ``cu_seqlens_k``: key offsets of a varlen
    batch whose key lengths differ from its query lengths. ``window_left`` /
    ``window_right``: query i sees keys i + delta - window_left ..
    i + delta + window_right (delta = Lk - Lq; -1: no bound; causal sets the
    right bound to 0). ``block_mask``: dense problems only, [Hm, ceil(Lq/bq),
    ceil(Lk/bk)] (Hm 1 or H; 2-D means Hm = 1) with ``block = (bq, bk)``; a
    zero entry drops that block of (query, key) pairs.
    ``rows``: optional query-row indices (per sequence) to evaluate; the other
    rows of the returned arrays are NaN.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu, cuk = _i32(cu_seqlens), _i32(cu_seqlens_k)
    if cuk is not None and cu is None:
        raise ValueError("cu_seqlens_k needs cu_seqlens")
    B, H, Hkv, Lq, Lk, d = _dims(q, k, cu, cuk)
    dv = _dv(v, k)
    bm, bmh, bq, bk = _block_mask(block_mask, H, Lq, Lk, block)
    o = np.full(q.shape[:-1] + (dv,), np.nan)
    lse = np.full((B, H, Lq) if cu is None else (H, q.shape[0]), np.nan)
    r = _i32(rows)
    rc = _load().oracle_fwd(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(o, _dp), _ptr(lse, _dp),
                            B, H, Hkv, Lq, Lk, d, dv, float(scale), int(bool(causal)),
                            int(window_left), int(window_right), _ptr(bm, _bp), bmh, bq, bk,
                            _ptr(cu, _ip), _ptr(cuk, _ip), _ptr(r, _ip), 0 if r is None else len(r),
                            nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_fwd failed with code {rc}")
    return o, lse


def bwd(q, k, v, dout, scale: float, causal: bool, cu_seqlens=None, qrows=None, krows=None,
        nthreads=None, cu_seqlens_k=None, window_left: int = -1, window_right: int = -1, block_mask=None,
        block=(128, 128)):
    """dQ, dK, dV of L = sum(O * dO) by the definition. Returns float64 arrays.

    ``qrows`` / ``krows``: optional row subsets for dQ / (dK, dV); other rows NaN.
    Pass an empty list to skip a group entirely.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu, cuk = _i32(cu_seqlens), _i32(cu_seqlens_k)
    if cuk is not None and cu is None:
        raise ValueError("cu_seqlens_k needs cu_seqlens")
    B, H, Hkv, Lq, Lk, d = _dims(q, k, cu, cuk)
    dvd = _dv(v, k)
    bm, bmh, bq, bk = _block_mask(block_mask, H, Lq, Lk, block)
    if dout.shape != q.shape[:-1] + (dvd,):
        raise ValueError("dout must have the rows and heads of q and the head dim of v")
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    qr, kr = _i32(qrows), _i32(krows)
    rc = _load().oracle_bwd(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(dout, _dp),
                            _ptr(dq, _dp), _ptr(dk, _dp), _ptr(dv, _dp),
                            B, H, Hkv, Lq, Lk, d, dvd, float(scale), int(bool(causal)),
                            int(window_left), int(window_right), _ptr(bm, _bp), bmh, bq, bk, _ptr(cu, _ip),
                            _ptr(cuk, _ip), _ptr(qr, _ip), 0 if qr is None else len(qr),
                            _ptr(kr, _ip), 0 if kr is None else len(kr),
                            nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_bwd failed with code {rc}")
    return dq, dk, dv
