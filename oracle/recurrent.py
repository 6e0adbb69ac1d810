"""ctypes front end of the C float64 token recurrence (test infrastructure).

The recurrence itself lives in ``kda_oracle.c``; this module only builds it on
first use and marshals numpy / torch-CPU arrays into it.
"""
import ctypes
import os

import numpy as np

from . import build as _build

DT_BF16, DT_F32, DT_F64 = 0, 1, 2

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.kda_oracle_run.restype = ctypes.c_int
        lib.kda_oracle_run.argtypes = [
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]
        lib.kda_oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().kda_oracle_threads())


def _as_buffer(x):
    """Return (numpy array, dtype code) without changing the stored bits."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach()
        if x.device.type != "cpu":
            raise ValueError("oracle inputs must live in host memory")
        x = x.contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), DT_BF16
        if x.dtype == torch.float32:
            return x.numpy(), DT_F32
        if x.dtype == torch.float64:
            return x.numpy(), DT_F64
        raise TypeError(f"unsupported dtype {x.dtype}")
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, DT_BF16
    if x.dtype == np.float32:
        return x, DT_F32
    if x.dtype == np.float64:
        return x, DT_F64
    raise TypeError(f"unsupported dtype {x.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def run(q, k, v, alpha, beta, cu_seqlens, start_pos=None, init_state=None,
        scale=1.0, want_output=True, want_final=True, snap_req=None,
        snap_interval=256, heads=None):
    """Token-by-token float64 KDA over a packed batch.

    Shapes: q, k [T, H, d_k]; v [T, H, d_v]; alpha [T, H, d_k]; beta [T, H];
    cu_seqlens int [n+1]; start_pos int [n] or None; init_state float64
    [n, H, d_k, d_v] or None.  q, k, v may be bf16 / fp32 / fp64 (same dtype);
    alpha and beta fp32 or fp64.  ``snap_req`` is a list of (seq, ordinal).
    ``heads`` = (h0, h1) restricts the work to heads h0 <= h < h1 (other heads of
    the outputs stay zero).

    Returns dict with ``o`` [T, H, d_v], ``final`` [n, H, d_k, d_v] and ``snaps``
    [len(snap_req), H, d_k, d_v] (float64; NaN where a requested snapshot was
    never reached).
    """
    lib = _load()
    qb, qdt = _as_buffer(q)
    kb, kdt = _as_buffer(k)
    vb, vdt = _as_buffer(v)
    if not (qdt == kdt == vdt):
        raise TypeError("q, k, v must share one dtype")
    ab, adt = _as_buffer(alpha)
    bb, bdt = _as_buffer(beta)
    if adt != bdt or adt == DT_BF16:
        raise TypeError("alpha and beta must both be fp32 or both fp64")
    T, H, d_k = qb.shape
    d_v = vb.shape[2]
    if kb.shape != (T, H, d_k) or vb.shape[:2] != (T, H) or ab.shape != (T, H, d_k) \
            or bb.shape != (T, H):
        raise ValueError("inconsistent shapes")
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    n = cu.shape[0] - 1
    if cu[0] != 0 or cu[-1] != T:
        raise ValueError("cu_seqlens must start at 0 and end at T")
    sp = None if start_pos is None else np.ascontiguousarray(np.asarray(start_pos, dtype=np.int32))
    init = None
    if init_state is not None:
        init = np.ascontiguousarray(np.asarray(init_state, dtype=np.float64))
        if init.shape != (n, H, d_k, d_v):
            raise ValueError("init_state shape")
    o = np.zeros((T, H, d_v), np.float64) if want_output else None
    fin = np.zeros((n, H, d_k, d_v), np.float64) if want_final else None
    req = np.zeros((0, 2), np.int32) if not snap_req else np.ascontiguousarray(
        np.asarray(snap_req, dtype=np.int32).reshape(-1, 2))
    snaps = np.full((req.shape[0], H, d_k, d_v), np.nan, np.float64)
    h0, h1 = (0, H) if heads is None else heads
    rc = lib.kda_oracle_run(
        n, H, d_k, d_v, qdt, _ptr(qb), _ptr(kb), _ptr(vb), adt, _ptr(ab), _ptr(bb),
        _ptr(cu), _ptr(sp), _ptr(init), float(scale), _ptr(o), _ptr(fin),
        int(snap_interval), int(req.shape[0]), _ptr(req) if req.shape[0] else None,
        _ptr(snaps) if req.shape[0] else None, int(h0), int(h1))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return {"o": o, "final": fin, "snaps": snaps}


__all__ = ["run", "threads", "DT_BF16", "DT_F32", "DT_F64"]

if os.environ.get("KDA_ORACLE_EAGER_BUILD"):
    _load()
