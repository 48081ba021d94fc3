"""CPU oracle for fused exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it.

All arithmetic is in fp64 in ``attn_oracle.c`` (plain loops, OpenMP over rows);
this module only marshals arrays.  Inputs may be torch tensors of any float
dtype (bf16 widens to fp64 exactly) or numpy arrays, laid out [B, H, S, D].
Outputs are numpy fp64 arrays.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None
_c_double_p = ctypes.POINTER(ctypes.c_double)
_c_i64_p = ctypes.POINTER(ctypes.c_int64)


def _bind(lib):
    i = ctypes.c_int
    d = ctypes.c_double
    p = ctypes.c_void_p
    lib.oracle_version.restype = i
    lib.oracle_max_threads.restype = i
    lib.oracle_set_threads.argtypes = [i]
    lib.oracle_fwd.argtypes = [p, p, p, i, i, i, i, i, i, i, d, p, p]
    lib.oracle_fwd.restype = i
    lib.oracle_fwd_rows.argtypes = [p, p, p, i, i, i, i, i, i, i, d, p, ctypes.c_int64, p, p]
    lib.oracle_fwd_rows.restype = i
    lib.oracle_bwd_units.argtypes = [p, p, p, p, i, i, i, i, i, i, i, d, p, ctypes.c_int64,
                                     p, p, p, p, p]
    lib.oracle_bwd_units.restype = i
    lib.oracle_fwd_mod.argtypes = [p, p, p, i, i, i, i, i, i, d, i, i, p, p, p, p]
    lib.oracle_fwd_mod.restype = i
    lib.oracle_fwd_rows_mod.argtypes = [p, p, p, i, i, i, i, i, i, d, i, i, p, p, p,
                                        ctypes.c_int64, p, p]
    lib.oracle_fwd_rows_mod.restype = i
    lib.oracle_bwd_units_mod.argtypes = [p, p, p, p, i, i, i, i, i, i, d, i, i, p, p, p,
                                         ctypes.c_int64, p, p, p, p, p]
    lib.oracle_bwd_units_mod.restype = i
    lib.oracle_fwd_mod_range.argtypes = [p, p, p, i, i, i, i, i, i, d, i, i, p, p, i, i, p, p]
    lib.oracle_fwd_mod_range.restype = i
    lib.oracle_lse_merge.argtypes = [p, p, i, ctypes.c_long, i, p, p]
    lib.oracle_lse_merge.restype = i
    for name in ("oracle_tiled_fwd_f64", "oracle_tiled_fwd_f32"):
        f = getattr(lib, name)
        f.argtypes = [p, p, p, i, i, i, i, i, i, i, d, i, i, i, d, p, p, p, p]
        f.restype = i
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle shared library."""
    global _LIB
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _LIB is None:
        _LIB = _bind(ctypes.CDLL(_build.build()))
    return _LIB


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: widen on the CPU (exact for bf16/fp16/fp32)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dims(q, k):
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    assert B == Bk and D == Dk, "q/k shape mismatch"
    return B, Hq, Hkv, Sq, Sk, D


def max_threads(lib=None) -> int:
    return (lib or load()).oracle_max_threads()


def set_threads(n: int, lib=None) -> None:
    (lib or load()).oracle_set_threads(int(n))


def fwd(q, k, v, causal: bool, scale: float, lib=None):
    """Plain-definition forward. Returns (O [B,Hq,Sq,D], LSE [B,Hq,Sq]) in fp64."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k)
    o = np.zeros((B, Hq, Sq, D))
    lse = np.zeros((B, Hq, Sq))
    rc = lib.oracle_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Sk, D, int(causal),
                        float(scale), _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_fwd rejected its arguments ({rc})")
    return o, lse


def fwd_rows(q, k, v, causal: bool, scale: float, rows, lib=None):
    """Forward for selected flat rows (b*Hq + h)*Sq + i. Returns (O [n,D], LSE [n])."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.zeros((len(rows), D))
    lse = np.zeros(len(rows))
    rc = lib.oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Sk, D, int(causal),
                             float(scale), _ptr(rows), len(rows), _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_fwd_rows rejected its arguments ({rc})")
    return o, lse


def bwd(q, k, v, do, causal: bool, scale: float, units=None, lib=None):
    """Textbook backward of the definition.

    ``units`` lists kv-head units b*Hkv + hk to compute (default: all).  Returns
    (dQ, dK, dV, O, LSE) at full size; slices outside the chosen units are NaN.
    """
    lib = lib or load()
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k)
    if units is None:
        units = np.arange(B * Hkv)
    units = np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    o = np.full(q.shape, np.nan)
    lse = np.full((B, Hq, Sq), np.nan)
    rc = lib.oracle_bwd_units(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, Hq, Hkv, Sq, Sk, D,
                              int(causal), float(scale), _ptr(units), len(units), _ptr(dq),
                              _ptr(dk), _ptr(dv), _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_bwd_units rejected its arguments ({rc})")
    return dq, dk, dv, o, lse


def _seqlens(seqlens_k, B):
    """Per-batch key lengths as a contiguous int32 array (None: all keys)."""
    if seqlens_k is None:
        return None
    if hasattr(seqlens_k, "detach"):
        seqlens_k = seqlens_k.detach().to("cpu").numpy()
    a = np.ascontiguousarray(np.asarray(seqlens_k, dtype=np.int32).reshape(-1))
    assert a.shape == (B,), "one key length per batch"
    return a


def _slopes(slopes, Hq):
    if slopes is None:
        return None
    a = _f64(slopes).reshape(-1)
    assert a.shape == (Hq,), "one slope per query head"
    return a


def fwd_mod(q, k, v, scale: float, window_left: int = -1, window_right: int = -1, slopes=None,
            seqlens_k=None, lib=None):
    """Forward with the score modification: key j visible to query i iff
    (window_left < 0 or j >= i - window_left) and (window_right < 0 or
    j <= i + window_right) and j < seqlens_k[b]; score scale*q.k +
    slopes[h]*(j - i).  Returns (O, LSE); a row with no visible key has O = 0,
    LSE = -inf."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k)
    sl = _slopes(slopes, Hq)
    sk = _seqlens(seqlens_k, B)
    o = np.zeros((B, Hq, Sq, D))
    lse = np.zeros((B, Hq, Sq))
    rc = lib.oracle_fwd_mod(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Sk, D, float(scale),
                            int(window_left), int(window_right),
                            None if sl is None else _ptr(sl), None if sk is None else _ptr(sk),
                            _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_fwd_mod rejected its arguments ({rc})")
    return o, lse


def fwd_rows_mod(q, k, v, scale: float, rows, window_left: int = -1, window_right: int = -1,
                 slopes=None, seqlens_k=None, lib=None):
    """fwd_mod for selected flat rows (b*Hq + h)*Sq + i. Returns (O [n,D], LSE [n])."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k)
    sl = _slopes(slopes, Hq)
    sk = _seqlens(seqlens_k, B)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.zeros((len(rows), D))
    lse = np.zeros(len(rows))
    rc = lib.oracle_fwd_rows_mod(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Sk, D, float(scale),
                                 int(window_left), int(window_right),
                                 None if sl is None else _ptr(sl),
                                 None if sk is None else _ptr(sk), _ptr(rows), len(rows),
                                 _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_fwd_rows_mod rejected its arguments ({rc})")
    return o, lse


def bwd_mod(q, k, v, do, scale: float, window_left: int = -1, window_right: int = -1,
            slopes=None, units=None, seqlens_k=None, lib=None):
    """Backward with the score modification (see fwd_mod); same return as bwd."""
    lib = lib or load()
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k)
    sl = _slopes(slopes, Hq)
    sk = _seqlens(seqlens_k, B)
    if units is None:
        units = np.arange(B * Hkv)
    units = np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    o = np.full(q.shape, np.nan)
    lse = np.full((B, Hq, Sq), np.nan)
    rc = lib.oracle_bwd_units_mod(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, Hq, Hkv, Sq, Sk, D,
                                  float(scale), int(window_left), int(window_right),
                                  None if sl is None else _ptr(sl),
                                  None if sk is None else _ptr(sk), _ptr(units), len(units),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_bwd_units_mod rejected its arguments ({rc})")
    return dq, dk, dv, o, lse


def fwd_mod_range(q, k, v, scale: float, k0: int, k1: int, window_left: int = -1,
                  window_right: int = -1, slopes=None, seqlens_k=None, lib=None):
    """fwd_mod over the keys [k0, k1) only (window and bias at the absolute key
    index).  Rows with no visible key there get O = 0, LSE = -inf."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k)
    sl = _slopes(slopes, Hq)
    sk = _seqlens(seqlens_k, B)
    o = np.zeros((B, Hq, Sq, D))
    lse = np.zeros((B, Hq, Sq))
    rc = lib.oracle_fwd_mod_range(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Sk, D, float(scale),
                                  int(window_left), int(window_right),
                                  None if sl is None else _ptr(sl),
                                  None if sk is None else _ptr(sk), int(k0), int(k1), _ptr(o),
                                  _ptr(lse))
    if rc:
        raise ValueError(f"oracle_fwd_mod_range rejected its arguments ({rc})")
    return o, lse


def lse_merge(o_parts, lse_parts, lib=None):
    """Merge n attention parts over disjoint key sets: o_parts [n, ..., D],
    lse_parts [n, ...] (natural log, -inf = empty part).  Returns (O, LSE)."""
    lib = lib or load()
    op = _f64(o_parts)
    lp = _f64(lse_parts)
    n, D = op.shape[0], op.shape[-1]
    assert lp.shape == op.shape[:-1], "one LSE per part row"
    rows = int(np.prod(lp.shape[1:], dtype=np.int64))
    o = np.zeros(op.shape[1:])
    lse = np.zeros(lp.shape[1:])
    rc = lib.oracle_lse_merge(_ptr(op), _ptr(lp), int(n), rows, int(D), _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_lse_merge rejected its arguments ({rc})")
    return o, lse


def tiled_fwd(q, k, v, causal: bool, scale: float, block_q: int = 64, block_kv: int = 64,
              mode: int = 0, threshold: float = 8.0, precision: str = "f64", lib=None):
    """Tiled online-softmax restatement (mode 0 always rescale, 1 threshold).

    Returns (O, LSE, n_rescaled, n_skipped).
    """
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Sq, Sk, D = _dims(q, k)
    o = np.zeros((B, Hq, Sq, D))
    lse = np.zeros((B, Hq, Sq))
    n_r = ctypes.c_int64(0)
    n_s = ctypes.c_int64(0)
    f = lib.oracle_tiled_fwd_f64 if precision == "f64" else lib.oracle_tiled_fwd_f32
    rc = f(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Sk, D, int(causal), float(scale),
           int(block_q), int(block_kv), int(mode), float(threshold), _ptr(o), _ptr(lse),
           ctypes.byref(n_r), ctypes.byref(n_s))
    if rc:
        raise ValueError(f"oracle tiled forward rejected its arguments ({rc})")
    return o, lse, n_r.value, n_s.value

