"""CPU float64 oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
import this package.  The CUDA library (exact_io_aware_35_gb300) never imports
it, and it never imports the CUDA library.

Two independent implementations of the same definition:
  * attn_oracle.c (through ctypes, OpenMP over rows) -- the oracle proper;
  * numpy_oracle.py -- whole-matrix numpy, used to cross-check the C one.

Inputs may be numpy arrays or CPU torch tensors of any float dtype; they are
converted exactly to float64 (bf16 -> f64 is exact).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import numpy_oracle  # noqa: F401  (re-exported)
from .build import LIB, build

_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_LL = ctypes.POINTER(ctypes.c_longlong)


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB)
        i = ctypes.c_int
        d = ctypes.c_double
        lib.oracle_attn_fwd.argtypes = [_D, _D, _D, _D, _D, i, i, i, i, i, i, d]
        lib.oracle_attn_fwd_rows.argtypes = [_D, _D, _D, _LL, i, _D, _D, i, i, i, i, i, i, d]
        lib.oracle_attn_bwd.argtypes = [_D, _D, _D, _D, _D, _D, _D, i, i, i, i, i, i, d]
        lib.oracle_attn_bwd_rows.argtypes = [_D, _D, _D, _D, _LL, i, _D, _LL, i, _D, _D,
                                             i, i, i, i, i, i, d]
        lib.oracle_attn_fwd_kv.argtypes = [_D, _D, _D, _D, _D, i, i, i, i, i, i, i, d]
        lib.oracle_attn_fwd_blockmask.argtypes = [_D, _D, _D, _D, _D, ctypes.c_void_p, i, i, i,
                                                  i, i, i, i, d]
        lib.oracle_attn_fwd_blockmask.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        for f in (lib.oracle_attn_fwd, lib.oracle_attn_fwd_rows, lib.oracle_attn_bwd,
                  lib.oracle_attn_bwd_rows, lib.oracle_attn_fwd_kv, lib.oracle_num_threads):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _shapes(q, k):
    if q.ndim != 4 or k.ndim != 4:
        raise ValueError("expected [B, N, H, d] arrays")
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape[0] != B or k.shape[1] != N or k.shape[3] != d or Hkv < 1 or Hq % Hkv:
        raise ValueError(f"incompatible shapes q{q.shape} k{k.shape}")
    return B, N, Hq, Hkv, d


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attn_fwd(q, k, v, causal: bool, scale: float):
    """Returns (o [B,N,Hq,d], lse [B,Hq,N]) in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, Hq, Hkv, d = _shapes(q, k)
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, N))
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 B, Hq, Hkv, N, d, int(bool(causal)), float(scale))
    if rc:
        raise RuntimeError(f"oracle_attn_fwd failed ({rc})")
    return o, lse


def attn_fwd_kv(q, k, v, causal: bool, scale: float):
    """Forward with Nq query rows against Nk keys (q [B,Nq,Hq,d], k, v
    [B,Nk,Hkv,d]); causal means query i sees keys j <= i + Nk - Nq (the
    queries are the sequence's last Nq positions).  Returns (o [B,Nq,Hq,d],
    lse [B,Hq,Nq]) in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or k.ndim != 4 or v.shape != k.shape:
        raise ValueError("expected [B, N, H, d] arrays")
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    if k.shape[0] != B or k.shape[3] != d or Hq % Hkv:
        raise ValueError(f"incompatible shapes q{q.shape} k{k.shape}")
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, Nq))
    rc = _load().oracle_attn_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                    Nq, Nk, d, int(bool(causal)), float(scale))
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_kv failed ({rc})")
    return o, lse


def attn_fwd_blockmask(q, k, v, block_mask, block: int, causal: bool, scale: float):
    """Forward under a block mask [Hq, nb, nb] (nonzero = the block is
    computed; nb = ceil(N / block)); rows with no visible key get O = 0 and
    lse = -inf.  Returns (o [B,N,Hq,d], lse [B,Hq,N]) in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, Hq, Hkv, d = _shapes(q, k)
    nb = (N + block - 1) // block
    mask = np.ascontiguousarray(np.asarray(block_mask).astype(np.uint8))
    if mask.shape != (Hq, nb, nb):
        raise ValueError(f"block mask shape {mask.shape}, expected {(Hq, nb, nb)}")
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, N))
    rc = _load().oracle_attn_fwd_blockmask(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                           mask.ctypes.data, int(block), B, Hq, Hkv, N, d,
                                           int(bool(causal)), float(scale))
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_blockmask failed ({rc})")
    return o, lse


def attn_fwd_rows(q, k, v, rows, causal: bool, scale: float):
    """Forward at query rows given as an [R, 3] array of (b, h, i).
    Returns (o_rows [R, d], lse_rows [R])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, Hq, Hkv, d = _shapes(q, k)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    R = rows.shape[0]
    o = np.zeros((R, d))
    lse = np.zeros(R)
    rc = _load().oracle_attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), rows.ctypes.data_as(_LL), R,
                                      _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                                      int(bool(causal)), float(scale))
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_rows failed ({rc})")
    return o, lse


def attn_bwd(q, k, v, dout, causal: bool, scale: float):
    """Returns (dq [B,N,Hq,d], dk [B,N,Hkv,d], dv [B,N,Hkv,d]) in float64."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, N, Hq, Hkv, d = _shapes(q, k)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rc = _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, Hq, Hkv, N, d, int(bool(causal)), float(scale))
    if rc:
        raise RuntimeError(f"oracle_attn_bwd failed ({rc})")
    return dq, dk, dv


def attn_bwd_rows(q, k, v, dout, qrows, kvrows, causal: bool, scale: float):
    """Backward at sampled rows.  qrows: [Rq, 3] (b, h, i) -> dq rows;
    kvrows: [Rk, 3] (b, hkv, j) -> dk, dv rows."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, N, Hq, Hkv, d = _shapes(q, k)
    qrows = np.ascontiguousarray(np.asarray(qrows, dtype=np.int64).reshape(-1, 3))
    kvrows = np.ascontiguousarray(np.asarray(kvrows, dtype=np.int64).reshape(-1, 3))
    dq = np.zeros((qrows.shape[0], d))
    dk = np.zeros((kvrows.shape[0], d))
    dv = np.zeros((kvrows.shape[0], d))
    rc = _load().oracle_attn_bwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                      qrows.ctypes.data_as(_LL), qrows.shape[0], _ptr(dq),
                                      kvrows.ctypes.data_as(_LL), kvrows.shape[0], _ptr(dk),
                                      _ptr(dv), B, Hq, Hkv, N, d, int(bool(causal)), float(scale))
    if rc:
        raise RuntimeError(f"oracle_attn_bwd_rows failed ({rc})")
    return dq, dk, dv
