"""Shared helpers for the GPU parity tests (CUDA path vs the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances: forward O max |dO| <= 2e-2, mean |dO| <= 2e-3, |dLSE| <= 1e-2;
# gradients max abs error <= 5e-2 * max |grad_ref|.
O_MAX, O_MEAN, LSE_MAX, GRAD_REL = 2e-2, 2e-3, 1e-2, 5e-2

SENTINEL_BF16 = 0x7FBF  # a NaN pattern no kernel writes
GUARD = 4096  # elements of guard band on each side


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def guarded_empty(shape, dtype, device):
    """Allocate a tensor inside a larger buffer whose margins hold a sentinel.
    Returns (view, buffer) -- check_guards(buffer, n) verifies the margins."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
    if dtype == torch.bfloat16:
        buf.view(torch.int16).fill_(SENTINEL_BF16)
    else:
        buf.fill_(float("nan"))
    view = buf[GUARD:GUARD + n].view(*shape)
    return view, buf


def check_guards(buf: torch.Tensor, n: int):
    head = buf[:GUARD]
    tail = buf[GUARD + n:]
    if buf.dtype == torch.bfloat16:
        assert bool((head.view(torch.int16) == SENTINEL_BF16).all()), "write before the output"
        assert bool((tail.view(torch.int16) == SENTINEL_BF16).all()), "write after the output"
    else:
        assert bool(torch.isnan(head).all()), "write before the output"
        assert bool(torch.isnan(tail).all()), "write after the output"


def assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    o = np64(o_gpu) if isinstance(o_gpu, torch.Tensor) else o_gpu
    lse = np64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    assert np.all(np.isfinite(lse)), f"{what}: non-finite LSE"
    d = np.abs(o - o_ref)
    dl = np.abs(lse - lse_ref)
    idx = np.unravel_index(np.argmax(d), d.shape)
    assert d.max() <= O_MAX, f"{what}: max|dO| {d.max():.3e} at {idx}"
    assert d.mean() <= O_MEAN, f"{what}: mean|dO| {d.mean():.3e}"
    assert dl.max() <= LSE_MAX, f"{what}: max|dLSE| {dl.max():.3e}"
    return float(d.max()), float(d.mean()), float(dl.max())


def assert_fwd_rows(o, lse, o_r, lse_r, what):
    """Rows the oracle leaves empty (LSE -inf) must be exactly O = 0, LSE = -inf;
    the others within the forward tolerance."""
    o, lse = np64(o), np64(lse)
    dead = np.isneginf(lse_r)
    assert np.array_equal(np.isneginf(lse), dead), f"{what}: rows with no key differ"
    assert np.all(o[dead] == 0.0), f"{what}: O of rows with no key"
    if (~dead).any():
        assert_fwd_close(o[~dead], lse[~dead], o_r[~dead], lse_r[~dead], what)
    return int(dead.sum())


def assert_grad_close(g_gpu, g_ref, what=""):
    g = np64(g_gpu) if isinstance(g_gpu, torch.Tensor) else g_gpu
    assert np.all(np.isfinite(g)), f"{what}: non-finite gradient"
    err = np.abs(g - g_ref)
    ref = np.abs(g_ref).max()
    idx = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= GRAD_REL * ref + 1e-6, (
        f"{what}: max err {err.max():.3e} > {GRAD_REL}*{ref:.3e} at {idx}")
    return float(err.max() / max(ref, 1e-30))
