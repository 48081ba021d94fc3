"""GB300 (sm_103a) fused exact attention: thin Python binding over libfa.so.

Every computation runs in the library's CUDA kernels; this module only checks
tensor properties, allocates outputs with torch and passes raw pointers plus the
current CUDA stream through the C ABI declared in ``include/fa.h``.  There is no
CPU or eager fallback: if the library is missing or a tensor is not a
contiguous bf16 CUDA tensor, the call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_OK = 0
FA_ERR_WORKSPACE = 4
FA_ERR_TIMEOUT = 6
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED",
                3: "FA_ERR_MISALIGNED", 4: "FA_ERR_WORKSPACE", 5: "FA_ERR_CUDA",
                6: "FA_ERR_TIMEOUT"}

#: every symbol include/fa.h declares
EXPORTS = ("fa_fwd", "fa_fwd_status", "fa_bwd_workspace_bytes", "fa_bwd", "fa_bwd_status",
           "fa_status_string", "fa_exp2_test", "fa_last_launch_count", "fa_set_timing_events",
           "fa_set_bwd_kernel",
           "fa_bwd_noalloc", "fa_fwd_mod", "fa_bwd_mod", "fa_fwd_split_count",
           "fa_fwd_split_workspace_bytes", "fa_fwd_split", "fa_lse_merge", "fa_wait_test",
           "fa_bwd_noalloc_status")


class ScoreMod(ctypes.Structure):
    """fa_score_mod: a sliding window (negative sides unbounded), optional
    per-head relative-position bias slopes and optional per-batch key counts
    (device pointers or None)."""
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("alibi_slopes", ctypes.c_void_p), ("seqlens_k", ctypes.c_void_p)]

_LIB = None


class FAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)}")
        self.code = code


def _bind(lib):
    vp, i, f, sz, i64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                         ctypes.c_int64)
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_status.argtypes = [vp]
    lib.fa_fwd_status.restype = i
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    lib.fa_bwd_workspace_bytes.restype = sz
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, sz, i,
                           vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_status.argtypes = [vp, vp]
    lib.fa_bwd_status.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_exp2_test.argtypes = [vp, vp, i64, i, vp]
    lib.fa_exp2_test.restype = i
    lib.fa_last_launch_count.argtypes = []
    lib.fa_last_launch_count.restype = i
    lib.fa_set_timing_events.argtypes = [vp, vp]
    lib.fa_set_timing_events.restype = i
    lib.fa_set_bwd_kernel.argtypes = [i, vp]
    lib.fa_set_bwd_kernel.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i,
                                   vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_noalloc_status.argtypes = [vp]
    lib.fa_bwd_noalloc_status.restype = i
    smp = ctypes.POINTER(ScoreMod)
    lib.fa_fwd_mod.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, smp, f, vp]
    lib.fa_fwd_mod.restype = i
    lib.fa_bwd_mod.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, smp, f, vp,
                               sz, i, vp]
    lib.fa_bwd_mod.restype = i
    lib.fa_fwd_split_count.argtypes = [i, i, i, i, i]
    lib.fa_fwd_split_count.restype = i
    lib.fa_fwd_split_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.fa_fwd_split_workspace_bytes.restype = sz
    lib.fa_fwd_split.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, smp, f, i, vp, sz, vp]
    lib.fa_fwd_split.restype = i
    lib.fa_lse_merge.argtypes = [vp, vp, i, vp, vp, i64, i, vp]
    lib.fa_lse_merge.restype = i
    lib.fa_wait_test.argtypes = [vp, i, vp, vp]
    lib.fa_wait_test.restype = i
    return lib


def _score_mod(causal, window, alibi_slopes, Hq, seqlens_k=None, B=None):
    """The fa_score_mod for a call, or None when the plain entry point applies."""
    if window is None and alibi_slopes is None and seqlens_k is None:
        return None
    wl, wr = (-1, 0 if causal else -1) if window is None else window
    if causal and window is not None:
        raise ValueError("give the causal mask as window=(-1, 0), not with causal=True")
    ptr = None
    if alibi_slopes is not None:
        if (not alibi_slopes.is_cuda or alibi_slopes.dtype != torch.float32
                or alibi_slopes.numel() != Hq or not alibi_slopes.is_contiguous()):
            raise TypeError("alibi_slopes must be a contiguous fp32 CUDA tensor of Hq slopes")
        ptr = alibi_slopes.data_ptr()
    lens = None
    if seqlens_k is not None:
        if (not seqlens_k.is_cuda or seqlens_k.dtype != torch.int32
                or seqlens_k.numel() != B or not seqlens_k.is_contiguous()):
            raise TypeError("seqlens_k must be a contiguous int32 CUDA tensor of B key counts")
        lens = seqlens_k.data_ptr()
    return ScoreMod(int(wl), int(wr), ptr, lens)


def lib():
    """The loaded libfa.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        _LIB = _bind(ctypes.CDLL(LIB_PATH))
    return _LIB


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous [B, H, S, D]")
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B, H, S, D]")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
        scale: float | None = None, out: torch.Tensor | None = None,
        lse: torch.Tensor | None = None, stream=None, window=None, alibi_slopes=None,
        n_splits: int | None = None, split_workspace: torch.Tensor | None = None,
        seqlens_k: torch.Tensor | None = None):
    """Forward attention. q [B,Hq,Sq,D], k/v [B,Hkv,Sk,D] bf16 CUDA.

    ``window=(left, right)``, ``alibi_slopes`` (fp32 [Hq]) and ``seqlens_k``
    (int32 [B] key counts: the key padding mask) select the score modification
    of fa_fwd_mod (include/fa.h); a row that sees no key gets O = 0, LSE = -inf.  ``n_splits`` (0: automatic)
    runs the split-KV form fa_fwd_split; its workspace is ``split_workspace``
    (uint8 CUDA) or allocated here.
    Returns (o [B,Hq,Sq,D] bf16, lse [B,Hq,Sq] fp32, natural log).
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    mod = _score_mod(causal, window, alibi_slopes, Hq, seqlens_k, B)
    if n_splits is not None:
        if mod is None and causal:
            mod = ScoreMod(-1, 0, None, None)
        ws_bytes = fwd_split_workspace_bytes(B, Hq, Sq, Sk, D, n_splits)
        if split_workspace is None:
            split_workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
        rc = lib().fa_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq,
                                Sk, D, None if mod is None else ctypes.byref(mod), float(scale),
                                int(n_splits), _ptr(split_workspace),
                                split_workspace.numel() * split_workspace.element_size(),
                                _stream(stream))
        if rc != FA_OK:
            raise FAError("fa_fwd_split", rc)
        return out, lse
    if mod is None:
        rc = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                          int(bool(causal)), float(scale), _stream(stream))
    else:
        rc = lib().fa_fwd_mod(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq,
                              Sk, D, ctypes.byref(mod), float(scale), _stream(stream))
    if rc != FA_OK:
        raise FAError("fa_fwd_mod" if mod is not None else "fa_fwd", rc)
    return out, lse


def fwd_split_count(B, Hq, Sq, Sk, sm_count: int = 0) -> int:
    """Splits fa_fwd_split uses for n_splits = 0 (sm_count 0: current device)."""
    return int(lib().fa_fwd_split_count(B, Hq, Sq, Sk, int(sm_count)))


def fwd_split_workspace_bytes(B, Hq, Sq, Sk, D, n_splits: int = 0) -> int:
    return int(lib().fa_fwd_split_workspace_bytes(B, Hq, Sq, Sk, D, int(n_splits)))


def lse_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out: torch.Tensor | None = None,
              lse: torch.Tensor | None = None, stream=None):
    """Log-sum-exp merge of parts over disjoint key sets (fa_lse_merge).

    o_parts [n, ..., D] fp32 and lse_parts [n, ...] fp32 (natural log, -inf for
    an empty part), contiguous CUDA.  Returns (o [..., D] bf16, lse [...] fp32).
    """
    for t, n in ((o_parts, "o_parts"), (lse_parts, "lse_parts")):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous fp32 CUDA tensor")
    if tuple(lse_parts.shape) != tuple(o_parts.shape[:-1]):
        raise ValueError("lse_parts must be o_parts' shape without the last dimension")
    n, D = o_parts.shape[0], o_parts.shape[-1]
    rows = lse_parts[0].numel() if n > 0 else 0
    if out is None:
        out = torch.empty(o_parts.shape[1:], dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    rc = lib().fa_lse_merge(_ptr(o_parts), _ptr(lse_parts), int(n), _ptr(out), _ptr(lse),
                            int(rows), int(D), _stream(stream))
    if rc != FA_OK:
        raise FAError("fa_lse_merge", rc)
    return out, lse


def bwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, deterministic=False) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, int(bool(deterministic))))


def bwd(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
        deterministic: bool = False, workspace: torch.Tensor | None = None,
        dq=None, dk=None, dv=None, stream=None, window=None, alibi_slopes=None,
        seqlens_k=None):
    """Backward attention. Returns (dq, dk, dv) bf16, same shapes as q, k, v.
    ``window`` / ``alibi_slopes`` / ``seqlens_k`` as in fwd (must match the
    forward call)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _check(t, n)
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise TypeError("lse must be a contiguous fp32 CUDA tensor")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = bwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, deterministic)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    mod = _score_mod(causal, window, alibi_slopes, Hq, seqlens_k, B)
    if mod is None:
        rc = lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                          _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Sk, D, int(bool(causal)),
                          float(scale), _ptr(workspace), workspace.numel(),
                          int(bool(deterministic)), _stream(stream))
    else:
        rc = lib().fa_bwd_mod(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Sk, D, ctypes.byref(mod),
                              float(scale), _ptr(workspace), workspace.numel(),
                              int(bool(deterministic)), _stream(stream))
    if rc != FA_OK:
        raise FAError("fa_bwd_mod" if mod is not None else "fa_bwd", rc)
    return dq, dk, dv


def fwd_status(stream=None) -> int:
    """Synchronise and return (then clear) the forward kernels' timeout record."""
    return int(lib().fa_fwd_status(_stream(stream)))


def bwd_status(workspace: torch.Tensor, stream=None) -> int:
    return int(lib().fa_bwd_status(_ptr(workspace), _stream(stream)))


def exp2_test(x: torch.Tensor, which: int, stream=None) -> torch.Tensor:
    """2^x through the kernel's MUFU path (which=0), polynomial path (which=1) or
    packed two-lane polynomial path (which=2)."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous fp32 CUDA tensor")
    y = torch.empty_like(x)
    rc = lib().fa_exp2_test(_ptr(x), _ptr(y), x.numel(), int(which), _stream(stream))
    if rc != FA_OK:
        raise FAError("fa_exp2_test", rc)
    return y


def wait_test(which: int, flag: torch.Tensor | None = None, stream=None) -> int:
    """Run one of the kernels' bounded waits (fa_wait_test); returns the status it
    wrote: FA_OK or FA_ERR_TIMEOUT (6).  flag: an int32 CUDA scalar for which=0."""
    status = torch.full((1,), -1, dtype=torch.int32, device=flag.device if flag is not None
                        else torch.device("cuda", torch.cuda.current_device()))
    rc = lib().fa_wait_test(None if flag is None else _ptr(flag), int(which), _ptr(status),
                            _stream(stream))
    if rc != FA_OK:
        raise FAError("fa_wait_test", rc)
    return int(status.item())


def last_launch_count() -> int:
    return int(lib().fa_last_launch_count())


def set_timing_events(start: "torch.cuda.Event | None", stop: "torch.cuda.Event | None") -> None:
    """Record ``start``/``stop`` around the main kernel of the next fwd/bwd call
    made by this thread (events must be created with timing enabled)."""
    for e in (start, stop):
        if e is not None and e.cuda_event == 0:
            e.record()  # torch creates the CUDA event lazily, on its first record
    ps = ctypes.c_void_p(start.cuda_event) if start is not None else None
    pe = ctypes.c_void_p(stop.cuda_event) if stop is not None else None
    rc = lib().fa_set_timing_events(ps, pe)
    if rc != FA_OK:
        raise FAError("fa_set_timing_events", rc)


BWD_KERNEL_AUTO, BWD_KERNEL_ONE_SM, BWD_KERNEL_PAIR = 0, 1, 2


def set_bwd_kernel(kind: int) -> int:
    """Backward main kernel for head dim 128, atomic dQ, no score modification
    (fa_set_bwd_kernel): BWD_KERNEL_AUTO, BWD_KERNEL_ONE_SM or BWD_KERNEL_PAIR
    (CTA pairs, 2-CTA MMA).  Returns the previous setting."""
    prev = ctypes.c_int(0)
    rc = lib().fa_set_bwd_kernel(int(kind), ctypes.byref(prev))
    if rc != FA_OK:
        raise FAError("fa_set_bwd_kernel", rc)
    return prev.value


class _Attention(torch.autograd.Function):
    """fwd in forward (saving O and LSE), bwd in backward; nothing else runs."""

    @staticmethod
    def forward(ctx, q, k, v, causal, scale, window, alibi_slopes, deterministic, seqlens_k):
        o, lse = fwd(q, k, v, causal=causal, scale=scale, window=window,
                     alibi_slopes=alibi_slopes, seqlens_k=seqlens_k)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.args = (causal, scale, window, alibi_slopes, deterministic, seqlens_k)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        causal, scale, window, alibi_slopes, deterministic, seqlens_k = ctx.args
        dq, dk, dv = bwd(q, k, v, o, do.contiguous(), lse, causal=causal, scale=scale,
                         deterministic=deterministic, window=window, alibi_slopes=alibi_slopes,
                         seqlens_k=seqlens_k)
        return dq, dk, dv, None, None, None, None, None, None


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
              scale: float | None = None, window=None, alibi_slopes=None,
              deterministic: bool = False, seqlens_k=None) -> torch.Tensor:
    """Exact attention as a differentiable op: O = softmax(scale q k^T + mods) v.

    q [B,Hq,Sq,D], k/v [B,Hkv,Sk,D] bf16 CUDA; ``causal``, ``window``,
    ``alibi_slopes`` and ``seqlens_k`` as in fwd; ``deterministic`` selects the
    backward mode.  O.backward() runs fa_bwd (the slopes get no gradient).
    Returns O bf16.
    """
    return _Attention.apply(q, k, v, causal, scale, window, alibi_slopes, deterministic,
                            seqlens_k)
