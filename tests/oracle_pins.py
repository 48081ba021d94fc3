"""Pins that tie the CPU oracle to facts other than itself.

Each ``pin_*`` takes a loaded oracle library and raises AssertionError when the
oracle disagrees with a closed form, an invariant, a hand-derived example, a
library routine on a special case, finite differences, or the harness printed
on the FlashAttention-4 pages.  ``test_oracle_pins.py`` runs them on the real
oracle; ``test_oracle_mutants.py`` runs them on deliberately broken copies of
the oracle source to show that each planted mistake is caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    assert err <= tol * scale, f"{what}: max err {err:.3e} > {tol:.1e} (scale {scale:.2f})"


def _parse(x):
    """'ln7' -> log(7), '11/7' -> 11/7, numbers pass through."""
    if isinstance(x, (int, float)):
        return float(x)
    x = x.strip()
    if x.startswith("ln"):
        return math.log(float(x[2:]))
    if "/" in x:
        a, b = x.split("/")
        return float(a) / float(b)
    return float(x)


# --------------------------------------------------------------------------- forward


def pin_hand_example(lib):
    """Exact fractions derived by hand (tests/golden/fwd_hand_example.json)."""
    g = json.load(open(os.path.join(GOLDEN, "fwd_hand_example.json")))
    q = np.array([[_parse(x) for x in row] for row in g["q"]])[None, None]
    k = np.array(g["k"], dtype=np.float64)[None, None]
    v = np.array(g["v"], dtype=np.float64)[None, None]
    for mode in ("noncausal", "causal"):
        o, lse = oracle.fwd(q, k, v, mode == "causal", g["scale"], lib=lib)
        o_ref = np.array([[_parse(x) for x in row] for row in g[mode]["o"]])
        lse_ref = np.array([_parse(x) for x in g[mode]["lse"]])
        _close(o[0, 0], o_ref, 1e-14, f"hand example O ({mode})")
        _close(lse[0, 0], lse_ref, 1e-14, f"hand example LSE ({mode})")


def pin_identical_keys(lib):
    """All keys equal: every allowed key has the same score, so O_i is the mean
    of the allowed values and LSE_i = scale q_i.k + ln(#allowed)."""
    rng = _rng(1)
    for causal in (False, True):
        B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 9, 13, 8
        q = _rand(rng, B, Hq, Sq, D)
        krow = _rand(rng, D)
        k = np.broadcast_to(krow, (B, Hkv, Sk, D)).copy()
        v = _rand(rng, B, Hkv, Sk, D)
        scale = 0.37
        o, lse = oracle.fwd(q, k, v, causal, scale, lib=lib)
        for b in range(B):
            for h in range(Hq):
                hk = h * Hkv // Hq
                for i in range(Sq):
                    n = min(i + 1, Sk) if causal else Sk
                    _close(o[b, h, i], v[b, hk, :n].mean(axis=0), 1e-12,
                           f"identical keys O causal={causal}")
                    _close(lse[b, h, i], scale * q[b, h, i] @ krow + math.log(n), 1e-12,
                           f"identical keys LSE causal={causal}")


def pin_causal_row0(lib):
    """Causal row 0 sees only key 0: O_0 = v_0 and LSE_0 = scale q_0.k_0."""
    rng = _rng(2)
    q = _rand(rng, 2, 3, 6, 16, std=3.0)
    k = _rand(rng, 2, 3, 6, 16, std=3.0)
    v = _rand(rng, 2, 3, 6, 16)
    o, lse = oracle.fwd(q, k, v, True, 0.25, lib=lib)
    _close(o[:, :, 0], v[:, :, 0], 1e-13, "causal row 0 O")
    _close(lse[:, :, 0], 0.25 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), 1e-13,
           "causal row 0 LSE")


def pin_scale_zero(lib):
    """scale = 0: uniform weights.  O = mean of allowed V rows, LSE = ln(#allowed)."""
    rng = _rng(3)
    q = _rand(rng, 1, 2, 7, 8)
    k = _rand(rng, 1, 2, 5, 8)
    v = _rand(rng, 1, 2, 5, 8)
    o, lse = oracle.fwd(q, k, v, False, 0.0, lib=lib)
    _close(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), 1e-13, "scale 0 O")
    _close(lse, np.full(lse.shape, math.log(5)), 1e-13, "scale 0 LSE")
    o, lse = oracle.fwd(q, k, v, True, 0.0, lib=lib)
    for i in range(7):
        n = min(i + 1, 5)
        _close(o[:, :, i], v[:, :, :n].mean(axis=2), 1e-13, "scale 0 causal O")
        _close(lse[:, :, i], np.full((1, 2), math.log(n)), 1e-13, "scale 0 causal LSE")


def pin_single_key(lib):
    """Sk = 1: softmax of one score is 1, so O = v_0 and LSE = the score."""
    rng = _rng(4)
    q = _rand(rng, 1, 2, 4, 8)
    k = _rand(rng, 1, 1, 1, 8)
    v = _rand(rng, 1, 1, 1, 8)
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, causal, 0.5, lib=lib)
        _close(o, np.broadcast_to(v[:, :1], o.shape), 1e-13, "single key O")
        _close(lse, 0.5 * np.einsum("bhid,bd->bhi", q, k[:, 0, 0]), 1e-13, "single key LSE")


def _library_attention(q, k, v, causal, scale):
    """scipy's logsumexp/softmax on scores formed with numpy: a special case that
    reduces attention to library routines (no shared code with the oracle)."""
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            hk = h * Hkv // Hq
            s = scale * (q[b, h] @ k[b, hk].T)
            if causal:
                s = np.where(np.arange(Sk)[None, :] <= np.arange(Sq)[:, None], s, -np.inf)
            lse[b, h] = scipy.special.logsumexp(s, axis=1)
            o[b, h] = scipy.special.softmax(s, axis=1) @ v[b, hk]
    return o, lse


def pin_library_routines(lib):
    """LSE equals scipy.special.logsumexp of the scores and O equals
    scipy.special.softmax(scores) @ V, including GQA, causal and Sq != Sk."""
    rng = _rng(5)
    for (B, Hq, Hkv, Sq, Sk, D, causal) in [(2, 4, 2, 17, 23, 8, False), (1, 6, 3, 19, 19, 16, True),
                                            (1, 2, 1, 11, 7, 4, True)]:
        q = _rand(rng, B, Hq, Sq, D, std=2.0)
        k = _rand(rng, B, Hkv, Sk, D, std=2.0)
        v = _rand(rng, B, Hkv, Sk, D)
        o, lse = oracle.fwd(q, k, v, causal, 0.3, lib=lib)
        o_ref, lse_ref = _library_attention(q, k, v, causal, 0.3)
        _close(o, o_ref, 1e-12, "O vs scipy softmax")
        _close(lse, lse_ref, 1e-12, "LSE vs scipy logsumexp")


def pin_softmax_rows_sum_to_one(lib):
    """With V = identity rows (Sk = D), O_i is the probability row P_i itself:
    it must be non-negative and sum to 1."""
    rng = _rng(6)
    Sk = D = 12
    q = _rand(rng, 1, 2, 9, D, std=2.0)
    k = _rand(rng, 1, 2, Sk, D, std=2.0)
    v = np.broadcast_to(np.eye(Sk), (1, 2, Sk, D)).copy()
    for causal in (False, True):
        o, _ = oracle.fwd(q, k, v, causal, 0.7, lib=lib)
        assert np.all(o >= -1e-15), "probabilities must be non-negative"
        _close(o.sum(axis=-1), np.ones(o.shape[:-1]), 1e-13, f"rows of P sum to 1 causal={causal}")
        if causal:
            for i in range(9):
                assert np.all(o[..., i, i + 1:] == 0), "causal: no weight on future keys"


def pin_key_permutation(lib):
    """Non-causal attention is invariant under a joint permutation of K and V rows."""
    rng = _rng(7)
    q = _rand(rng, 1, 2, 10, 8)
    k = _rand(rng, 1, 2, 21, 8)
    v = _rand(rng, 1, 2, 21, 8)
    perm = rng.permutation(21)
    o1, l1 = oracle.fwd(q, k, v, False, 0.4, lib=lib)
    o2, l2 = oracle.fwd(q, k[:, :, perm], v[:, :, perm], False, 0.4, lib=lib)
    _close(o1, o2, 1e-13, "permutation O")
    _close(l1, l2, 1e-13, "permutation LSE")


def pin_gqa_equals_repeated_mha(lib):
    """Grouped heads equal plain multi-head attention with each kv head repeated
    Hq/Hkv times (contiguous groups)."""
    rng = _rng(8)
    B, Hq, Hkv, S, D = 2, 8, 2, 12, 8
    q = _rand(rng, B, Hq, S, D)
    k = _rand(rng, B, Hkv, S, D)
    v = _rand(rng, B, Hkv, S, D)
    kr = np.repeat(k, Hq // Hkv, axis=1)
    vr = np.repeat(v, Hq // Hkv, axis=1)
    for causal in (False, True):
        o1, l1 = oracle.fwd(q, k, v, causal, 0.3, lib=lib)
        o2, l2 = oracle.fwd(q, kr, vr, causal, 0.3, lib=lib)
        _close(o1, o2, 1e-14, "GQA O")
        _close(l1, l2, 1e-14, "GQA LSE")


def pin_rows_match_full(lib):
    """The sampled-row entry point agrees with the full forward."""
    rng = _rng(9)
    q = _rand(rng, 2, 4, 9, 8)
    k = _rand(rng, 2, 2, 11, 8)
    v = _rand(rng, 2, 2, 11, 8)
    o, lse = oracle.fwd(q, k, v, True, 0.5, lib=lib)
    rows = [0, 5, 17, 40, 71]
    o_r, l_r = oracle.fwd_rows(q, k, v, True, 0.5, rows, lib=lib)
    _close(o_r, o.reshape(-1, 8)[rows], 0.0, "rows O")
    _close(l_r, lse.reshape(-1)[rows], 0.0, "rows LSE")


def pin_pages_harness(lib):
    """The pages' validation harness: seed 42, B=2, H=4, S=256, D=128 fp32 normal
    inputs; the tiled loop (64x64 blocks, rescale every tile) must match the plain
    softmax definition with cosine similarity > 0.9999 -- and in fp64 it is
    exact to rounding."""
    g = json.load(open(os.path.join(GOLDEN, "pages_harness.json")))
    torch.manual_seed(g["seed"])
    shape = (g["batch"], g["heads"], g["seq_len"], g["head_dim"])
    q = torch.randn(*shape)
    k = torch.randn(*shape)
    v = torch.randn(*shape)
    scale = 1.0 / math.sqrt(g["head_dim"])
    o_plain, lse_plain = oracle.fwd(q, k, v, g["causal"], scale, lib=lib)
    for prec, tol in (("f64", 1e-12), ("f32", 2e-5)):
        o_t, lse_t, _, _ = oracle.tiled_fwd(q, k, v, g["causal"], scale, g["block_q"],
                                            g["block_kv"], mode=0, precision=prec, lib=lib)
        a, b = o_t.ravel(), o_plain.ravel()
        cos = float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))
        assert cos > g["min_cosine_similarity"], f"harness cosine {cos}"
        _close(o_t, o_plain, tol, f"harness tiled O ({prec})")
        _close(lse_t, lse_plain, tol, f"harness tiled LSE ({prec})")
    # the library special case on the same inputs
    o_lib, _ = _library_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                  False, scale)
    _close(o_plain, o_lib, 1e-12, "harness plain vs scipy")


def _spiky(rng, B, Hq, Hkv, S, D):
    q = _rand(rng, B, Hq, S, D, std=3.0)
    k = _rand(rng, B, Hkv, S, D, std=3.0)
    for b in range(B):
        for h in range(Hkv):
            rows = rng.choice(S, size=max(1, S // 20), replace=False)
            k[b, h, rows] *= 8.0
    v = _rand(rng, B, Hkv, S, D)
    return q, k, v


def pin_conditional_rescale(lib):
    """The threshold variant (skip the rescale unless the running max grows by
    more than 8 in log2 units) equals the plain definition, on inputs with large
    late maxima, for several tile shapes; the rescale both fires and is skipped."""
    rng = _rng(10)
    q, k, v = _spiky(rng, 1, 4, 2, 300, 16)
    scale = 0.25
    for causal in (False, True):
        o_ref, lse_ref = oracle.fwd(q, k, v, causal, scale, lib=lib)
        for bq, bk in ((128, 128), (64, 32), (17, 50)):
            o_t, lse_t, n_r, n_s = oracle.tiled_fwd(q, k, v, causal, scale, bq, bk, mode=1,
                                                    threshold=8.0, lib=lib)
            _close(o_t, o_ref, 1e-12, f"threshold tiled O {bq}x{bk}")
            _close(lse_t, lse_ref, 1e-12, f"threshold tiled LSE {bq}x{bk}")
            assert n_r > 0, "rescale never fired"
            assert n_s > 0, "rescale never skipped"
            o0, lse0, _, _ = oracle.tiled_fwd(q, k, v, causal, scale, bq, bk, mode=0, lib=lib)
            _close(o0, o_ref, 1e-12, f"always-rescale tiled O {bq}x{bk}")
            _close(lse0, lse_ref, 1e-12, f"always-rescale tiled LSE {bq}x{bk}")
        o32, lse32, _, _ = oracle.tiled_fwd(q, k, v, causal, scale, 128, 128, mode=1,
                                            precision="f32", lib=lib)
        _close(o32, o_ref, 1e-4, "threshold tiled fp32 O")
        _close(lse32, lse_ref, 1e-4, "threshold tiled fp32 LSE")


def pin_threshold_extremes(lib):
    """Threshold 0 rescales whenever the max grows; a huge threshold never
    rescales after the first tile (it overflows only if scores span > 2^128,
    which these inputs do not).  Both still equal the definition."""
    rng = _rng(11)
    q = _rand(rng, 1, 2, 64, 8)
    k = _rand(rng, 1, 2, 96, 8)
    v = _rand(rng, 1, 2, 96, 8)
    o_ref, lse_ref = oracle.fwd(q, k, v, False, 0.5, lib=lib)
    o_t, lse_t, n_r, n_s = oracle.tiled_fwd(q, k, v, False, 0.5, 16, 16, mode=1, threshold=0.0,
                                            lib=lib)
    assert n_s == 0 and n_r > 0
    _close(o_t, o_ref, 1e-12, "threshold 0 O")
    o_t, lse_t, n_r, n_s = oracle.tiled_fwd(q, k, v, False, 0.5, 16, 16, mode=1, threshold=1e9,
                                            lib=lib)
    assert n_r == 0 and n_s > 0
    _close(o_t, o_ref, 1e-12, "threshold inf O")
    _close(lse_t, lse_ref, 1e-12, "threshold inf LSE")


# --------------------------------------------------------------------------- backward


def _loss(q, k, v, do, causal, scale, lib):
    o, _ = oracle.fwd(q, k, v, causal, scale, lib=lib)
    return float(np.sum(do * o))


def pin_bwd_finite_differences(lib):
    """Central differences (h = 1e-6, fp64) of L = sum(dO * O) against dQ, dK, dV,
    for MHA and GQA, causal and not."""
    rng = _rng(12)
    h = 1e-6
    for (B, Hq, Hkv, Sq, Sk, D, causal) in [(1, 1, 1, 4, 4, 4, False), (1, 2, 1, 8, 8, 4, True),
                                            (1, 2, 2, 5, 8, 8, True), (1, 4, 2, 6, 5, 4, False)]:
        q = _rand(rng, B, Hq, Sq, D)
        k = _rand(rng, B, Hkv, Sk, D)
        v = _rand(rng, B, Hkv, Sk, D)
        do = _rand(rng, B, Hq, Sq, D)
        scale = 0.6
        dq, dk, dv, _, _ = oracle.bwd(q, k, v, do, causal, scale, lib=lib)
        for name, x, g in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
            num = np.zeros_like(x)
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                xp = x.copy()
                xp[idx] += h
                xm = x.copy()
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = {"q": q, "k": k, "v": v}
                key = {"dQ": "q", "dK": "k", "dV": "v"}[name]
                args_p[key] = xp
                args_m[key] = xm
                num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, causal, scale, lib)
                            - _loss(args_m["q"], args_m["k"], args_m["v"], do, causal, scale,
                                    lib)) / (2 * h)
            err = np.max(np.abs(num - g))
            ref = max(np.max(np.abs(num)), 1e-3)
            assert err <= 1e-6 * ref + 1e-9, f"{name} finite differences: {err:.3e} (ref {ref:.3e})"


def pin_bwd_invariants(lib):
    """sum_j dS_ij = 0 for every row, so sum_j dK_j = 0 per kv head; and since
    rows of P sum to 1, sum_j dV_j = sum_i dO_i over the group's q heads."""
    rng = _rng(13)
    B, Hq, Hkv, S, D = 2, 4, 2, 33, 8
    q = _rand(rng, B, Hq, S, D, std=2.0)
    k = _rand(rng, B, Hkv, S, D, std=2.0)
    v = _rand(rng, B, Hkv, S, D)
    do = _rand(rng, B, Hq, S, D)
    for causal in (False, True):
        dq, dk, dv, o, lse = oracle.bwd(q, k, v, do, causal, 0.4, lib=lib)
        _close(dk.sum(axis=2), np.zeros((B, Hkv, D)), 1e-12, "sum_j dK_j = 0")
        g = Hq // Hkv
        do_sum = do.reshape(B, Hkv, g, S, D).sum(axis=(2, 3))
        _close(dv.sum(axis=2), do_sum, 1e-12, "sum_j dV_j = sum_i dO_i")
        o2, lse2 = oracle.fwd(q, k, v, causal, 0.4, lib=lib)
        _close(o, o2, 1e-14, "bwd's own forward O")
        _close(lse, lse2, 1e-14, "bwd's own forward LSE")


def pin_bwd_closed_forms(lib):
    """Sk = 1: P = 1 so dS = 0 -> dQ = dK = 0 and dV_0 = sum_i dO_i.
    scale = 0: dQ = dK = 0 and dV_j = sum_{i allowed to see j} dO_i / n_i."""
    rng = _rng(14)
    q = _rand(rng, 1, 2, 6, 4)
    do = _rand(rng, 1, 2, 6, 4)
    k1 = _rand(rng, 1, 1, 1, 4)
    v1 = _rand(rng, 1, 1, 1, 4)
    dq, dk, dv, _, _ = oracle.bwd(q, k1, v1, do, False, 0.9, lib=lib)
    _close(dq, np.zeros_like(dq), 1e-14, "Sk=1 dQ")
    _close(dk, np.zeros_like(dk), 1e-14, "Sk=1 dK")
    _close(dv[0, 0, 0], do[0].sum(axis=(0, 1)), 1e-13, "Sk=1 dV")
    k = _rand(rng, 1, 1, 6, 4)
    v = _rand(rng, 1, 1, 6, 4)
    dq, dk, dv, _, _ = oracle.bwd(q, k, v, do, True, 0.0, lib=lib)
    _close(dq, np.zeros_like(dq), 1e-14, "scale 0 dQ")
    _close(dk, np.zeros_like(dk), 1e-14, "scale 0 dK")
    expect = np.zeros((6, 4))
    for j in range(6):
        for i in range(j, 6):
            expect[j] += do[0, :, i].sum(axis=0) / (i + 1)
    _close(dv[0, 0], expect, 1e-13, "scale 0 causal dV")


# ------------------------------------------------------------- score modification


def _mask(Sq, Sk, wl, wr):
    """Dense visibility matrix of the sliding window, built by comparison."""
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    m = np.ones((Sq, Sk), dtype=bool)
    if wl >= 0:
        m &= j >= i - wl
    if wr >= 0:
        m &= j <= i + wr
    return m


def pin_mod_window_zero(lib):
    """A window of zero on both sides: query i sees key i alone, so O_i = v_i and
    LSE_i = scale * q_i . k_i (the bias is zero at j = i)."""
    rng = _rng(21)
    q = _rand(rng, 1, 2, 7, 4)
    k = _rand(rng, 1, 2, 7, 4)
    v = _rand(rng, 1, 2, 7, 4)
    o, lse = oracle.fwd_mod(q, k, v, 0.7, 0, 0, slopes=[0.3, -1.1], lib=lib)
    _close(o, v, 1e-14, "window 0: O = V")
    _close(lse, 0.7 * np.einsum("bhsd,bhsd->bhs", q, k), 1e-13, "window 0: LSE")


def pin_mod_alibi_identical_keys(lib):
    """All keys equal: the score is c + a*(j - i), so over the visible keys
    lo..hi-1 the weights are a geometric sequence: LSE_i = c - a*i +
    log(e^(a*lo) (e^(a*n) - 1) / (e^a - 1)) and O_i = sum_j w_j v_j."""
    rng = _rng(22)
    D, Sq, Sk = 4, 9, 11
    q = _rand(rng, 1, 1, Sq, D)
    kk = _rand(rng, D)
    k = np.broadcast_to(kk, (1, 1, Sk, D)).copy()
    v = _rand(rng, 1, 1, Sk, D)
    a, scale, wl, wr = 0.45, 0.8, 3, 2
    o, lse = oracle.fwd_mod(q, k, v, scale, wl, wr, slopes=[a], lib=lib)
    for i in range(Sq):
        lo, hi = max(0, i - wl), min(Sk, i + wr + 1)
        n = hi - lo
        c = scale * float(q[0, 0, i] @ kk)
        geo = math.exp(a * lo) * math.expm1(a * n) / math.expm1(a)
        assert abs(lse[0, 0, i] - (c - a * i + math.log(geo))) < 1e-12, f"alibi LSE row {i}"
        w = np.exp(a * np.arange(lo, hi)) / geo
        _close(o[0, 0, i], w @ v[0, 0, lo:hi], 1e-13, f"alibi O row {i}")


def pin_mod_dense_brute_force(lib):
    """A dense score matrix with the bias added and invisible pairs set to -inf,
    reduced with scipy's logsumexp: LSE and O on random inputs, GQA."""
    rng = _rng(23)
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 10, 13, 5
    q = _rand(rng, B, Hq, Sq, D)
    k = _rand(rng, B, Hkv, Sk, D)
    v = _rand(rng, B, Hkv, Sk, D)
    slopes = np.array([0.2, -0.5, 1.3, 0.0])
    for wl, wr in ((4, 1), (-1, 2), (3, -1), (12, 0)):
        o, lse = oracle.fwd_mod(q, k, v, 0.9, wl, wr, slopes=slopes, lib=lib)
        vis = _mask(Sq, Sk, wl, wr)
        rel = np.arange(Sk)[None, :] - np.arange(Sq)[:, None]
        for h in range(Hq):
            hk = h * Hkv // Hq
            sc = 0.9 * q[0, h] @ k[0, hk].T + slopes[h] * rel
            sc = np.where(vis, sc, -np.inf)
            ref_lse = scipy.special.logsumexp(sc, axis=1)
            _close(lse[0, h], ref_lse, 1e-12, f"dense LSE wl={wl} wr={wr} h={h}")
            _close(o[0, h], np.exp(sc - ref_lse[:, None]) @ v[0, hk], 1e-12,
                   f"dense O wl={wl} wr={wr} h={h}")


def pin_mod_reduces_to_plain(lib):
    """No window and no bias is the plain definition; window (-1, 0) is the causal
    one; the row-selected form matches the full one."""
    rng = _rng(24)
    q = _rand(rng, 2, 2, 9, 6)
    k = _rand(rng, 2, 1, 9, 6)
    v = _rand(rng, 2, 1, 9, 6)
    for wr, causal in ((-1, False), (0, True)):
        o, lse = oracle.fwd_mod(q, k, v, 0.5, -1, wr, lib=lib)
        o2, lse2 = oracle.fwd(q, k, v, causal, 0.5, lib=lib)
        _close(o, o2, 1e-14, f"mod O vs plain (causal={causal})")
        _close(lse, lse2, 1e-14, f"mod LSE vs plain (causal={causal})")
    rows = [0, 5, 17, 35]
    o, lse = oracle.fwd_mod(q, k, v, 0.5, 2, 3, slopes=[0.7, -0.2], lib=lib)
    orow, lrow = oracle.fwd_rows_mod(q, k, v, 0.5, rows, 2, 3, slopes=[0.7, -0.2], lib=lib)
    _close(orow, o.reshape(-1, 6)[rows], 1e-15, "mod rows vs full O")
    _close(lrow, lse.reshape(-1)[rows], 1e-15, "mod rows vs full LSE")


def _loss_mod(q, k, v, do, scale, wl, wr, slopes, lib):
    o, _ = oracle.fwd_mod(q, k, v, scale, wl, wr, slopes=slopes, lib=lib)
    return float(np.sum(do * o))


def pin_mod_bwd_finite_differences(lib):
    """Central differences (h = 1e-6, fp64) of L = sum(dO * O) under a window and
    a bias, against the modified backward."""
    rng = _rng(25)
    h = 1e-6
    for (Hq, Hkv, Sq, Sk, D, wl, wr, slopes) in [(2, 1, 7, 8, 4, 2, 1, [0.6, -0.4]),
                                                 (1, 1, 6, 6, 4, -1, 0, [0.9])]:
        q = _rand(rng, 1, Hq, Sq, D)
        k = _rand(rng, 1, Hkv, Sk, D)
        v = _rand(rng, 1, Hkv, Sk, D)
        do = _rand(rng, 1, Hq, Sq, D)
        dq, dk, dv, _, _ = oracle.bwd_mod(q, k, v, do, 0.6, wl, wr, slopes=slopes, lib=lib)
        for key, g in (("q", dq), ("k", dk), ("v", dv)):
            x = {"q": q, "k": k, "v": v}[key]
            num = np.zeros_like(x)
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                args = []
                for sgn in (1, -1):
                    xs = x.copy()
                    xs[idx] += sgn * h
                    a = {"q": q, "k": k, "v": v}
                    a[key] = xs
                    args.append(_loss_mod(a["q"], a["k"], a["v"], do, 0.6, wl, wr, slopes, lib))
                num[idx] = (args[0] - args[1]) / (2 * h)
            err = np.max(np.abs(num - g))
            ref = max(np.max(np.abs(num)), 1e-3)
            assert err <= 1e-6 * ref + 1e-9, f"mod d{key} finite differences: {err:.3e}"


def pin_mod_bwd_invariants(lib):
    """Rows of P still sum to one under a window and a bias: sum_j dK_j = 0 and
    sum_j dV_j = sum_i dO_i over the group."""
    rng = _rng(26)
    B, Hq, Hkv, S, D = 1, 2, 1, 21, 6
    q = _rand(rng, B, Hq, S, D, std=1.5)
    k = _rand(rng, B, Hkv, S, D, std=1.5)
    v = _rand(rng, B, Hkv, S, D)
    do = _rand(rng, B, Hq, S, D)
    dq, dk, dv, _, _ = oracle.bwd_mod(q, k, v, do, 0.5, 5, 3, slopes=[0.8, -0.3], lib=lib)
    _close(dk.sum(axis=2), np.zeros((B, Hkv, D)), 1e-12, "mod sum_j dK_j = 0")
    _close(dv.sum(axis=2), do.sum(axis=(1, 2)).reshape(B, Hkv, D), 1e-12,
           "mod sum_j dV_j = sum_i dO_i")


def pin_mod_key_padding(lib):
    """Per-batch key lengths: batch b with L_b keys gives what the same problem
    gives with K and V cut to their first L_b rows (window and bias keep the
    absolute indices, so the cut changes nothing else); L_b = 0 gives O = 0 and
    LSE = -inf; a length above Sk is Sk.  The backward: gradients of the cut
    problem on the kept keys, dK = dV = 0 past L_b, and dQ = 0 for rows that see
    no key."""
    rng = _rng(27)
    B, Hq, Hkv, Sq, Sk, D = 4, 2, 1, 9, 11, 4
    q = _rand(rng, B, Hq, Sq, D, std=1.5)
    k = _rand(rng, B, Hkv, Sk, D, std=1.5)
    v = _rand(rng, B, Hkv, Sk, D)
    do = _rand(rng, B, Hq, Sq, D)
    lens = np.array([7, 0, 11, 40], dtype=np.int32)
    slopes = [0.4, -0.9]
    for wl, wr in ((3, 1), (-1, -1), (-1, 0)):
        o, lse = oracle.fwd_mod(q, k, v, 0.7, wl, wr, slopes=slopes, seqlens_k=lens, lib=lib)
        dq, dk, dv, o2, lse2 = oracle.bwd_mod(q, k, v, do, 0.7, wl, wr, slopes=slopes,
                                              seqlens_k=lens, lib=lib)
        _close(o2, o, 0.0, f"padding bwd O = fwd O ({wl},{wr})")
        for b in range(B):
            L = min(int(lens[b]), Sk)
            tag = f"padding b={b} L={L} window ({wl},{wr})"
            if L == 0:
                assert np.all(o[b] == 0.0) and np.all(np.isneginf(lse[b])), tag + ": empty"
                assert np.all(dq[b] == 0.0) and np.all(dk[b] == 0.0) and np.all(dv[b] == 0.0)
                continue
            sl = (slice(b, b + 1), slice(None), slice(0, L))
            oc, lc = oracle.fwd_mod(q[b:b + 1], k[sl], v[sl], 0.7, wl, wr, slopes=slopes, lib=lib)
            _close(o[b:b + 1], oc, 1e-15, tag + ": O")
            _close(lse[b:b + 1], lc, 1e-15, tag + ": LSE")
            gq, gk, gv, _, _ = oracle.bwd_mod(q[b:b + 1], k[sl], v[sl], do[b:b + 1], 0.7, wl, wr,
                                              slopes=slopes, lib=lib)
            _close(dq[b:b + 1], gq, 1e-15, tag + ": dQ")
            _close(dk[sl], gk, 1e-15, tag + ": dK")
            _close(dv[sl], gv, 1e-15, tag + ": dV")
            assert np.all(dk[b, :, L:] == 0.0) and np.all(dv[b, :, L:] == 0.0), tag + ": tail"
        # the key-range form with lengths merges back to the full result
        parts = [oracle.fwd_mod_range(q, k, v, 0.7, a, c, wl, wr, slopes=slopes,
                                      seqlens_k=lens, lib=lib) for a, c in ((0, 4), (4, 11))]
        om, lm = oracle.lse_merge(np.stack([p[0] for p in parts]),
                                  np.stack([p[1] for p in parts]), lib=lib)
        _close(om, o, 1e-12, f"padding merged O ({wl},{wr})")
        live = np.isfinite(lse)
        assert np.array_equal(np.isneginf(lm), ~live), f"padding merged empty rows ({wl},{wr})"
        _close(lm[live], lse[live], 1e-12, f"padding merged LSE ({wl},{wr})")
    rows = [0, Sq + 3, 2 * Hq * Sq - 1, 3 * Hq * Sq + 5]
    orow, lrow = oracle.fwd_rows_mod(q, k, v, 0.7, rows, 3, 1, slopes=slopes, seqlens_k=lens,
                                     lib=lib)
    o, lse = oracle.fwd_mod(q, k, v, 0.7, 3, 1, slopes=slopes, seqlens_k=lens, lib=lib)
    _close(orow, o.reshape(-1, D)[rows], 0.0, "padding rows O")
    assert np.array_equal(lrow, lse.reshape(-1)[rows]), "padding rows LSE"


# --------------------------------------------------------------------------- split-KV


def pin_split_partition(lib):
    """The softmax over a union of disjoint key sets: the parts over any
    partition of [0, Sk), merged, give the full attention (window, bias, GQA,
    ragged chunks, rows with no visible key in some chunks)."""
    rng = _rng(31)
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 19, 23, 5
    q = _rand(rng, B, Hq, Sq, D, std=1.5)
    k = _rand(rng, B, Hkv, Sk, D, std=1.5)
    v = _rand(rng, B, Hkv, Sk, D)
    slopes = np.array([0.3, -0.7, 0.0, 1.1])
    cuts = [0, 5, 6, 17, 23]
    for wl, wr, sl in ((4, 2, slopes), (-1, 0, None), (-1, -1, None), (6, -1, slopes)):
        o, lse = oracle.fwd_mod(q, k, v, 0.8, wl, wr, slopes=sl, lib=lib)
        parts = [oracle.fwd_mod_range(q, k, v, 0.8, a, b, wl, wr, slopes=sl, lib=lib)
                 for a, b in zip(cuts[:-1], cuts[1:])]
        if wl == 4:
            assert any(np.isneginf(p[1]).any() for p in parts), "some rows empty in a chunk"
        om, lm = oracle.lse_merge(np.stack([p[0] for p in parts]),
                                  np.stack([p[1] for p in parts]), lib=lib)
        _close(om, o, 1e-12, f"merged O wl={wl} wr={wr}")
        _close(lm, lse, 1e-12, f"merged LSE wl={wl} wr={wr}")


def pin_split_range_special_cases(lib):
    """The whole key range is the unrestricted forward; an empty range gives
    O = 0 and LSE = -inf; a one-key range gives O = v_j and LSE = the score of
    (i, j) where j is visible, and the empty result where it is not."""
    rng = _rng(32)
    Sq, Sk, D = 8, 9, 4
    q = _rand(rng, 1, 1, Sq, D)
    k = _rand(rng, 1, 1, Sk, D)
    v = _rand(rng, 1, 1, Sk, D)
    wl, wr, a, scale = 2, 1, 0.4, 0.9
    o, lse = oracle.fwd_mod(q, k, v, scale, wl, wr, slopes=[a], lib=lib)
    o2, lse2 = oracle.fwd_mod_range(q, k, v, scale, 0, Sk, wl, wr, slopes=[a], lib=lib)
    _close(o2, o, 0.0, "range [0, Sk) O")
    _close(lse2, lse, 0.0, "range [0, Sk) LSE")
    o3, lse3 = oracle.fwd_mod_range(q, k, v, scale, 3, 3, wl, wr, slopes=[a], lib=lib)
    assert np.all(o3 == 0.0) and np.all(np.isneginf(lse3)), "empty range"
    j = 4
    o4, lse4 = oracle.fwd_mod_range(q, k, v, scale, j, j + 1, wl, wr, slopes=[a], lib=lib)
    for i in range(Sq):
        if i - wl <= j <= i + wr:
            _close(o4[0, 0, i], v[0, 0, j], 1e-15, f"one key O row {i}")
            ref = scale * float(q[0, 0, i] @ k[0, 0, j]) + a * (j - i)
            assert abs(lse4[0, 0, i] - ref) < 1e-13, f"one key LSE row {i}"
        else:
            assert np.all(o4[0, 0, i] == 0.0) and np.isneginf(lse4[0, 0, i]), f"hidden row {i}"


def pin_merge_closed_forms(lib):
    """Merge weights by hand: one part is the identity; two parts with equal LSE
    average with LSE + ln 2; LSEs ln 3 apart weigh 3/4 and 1/4 (also near
    LSE = 1000, where exp overflows without the max shift); an empty part
    (-inf) is ignored; all parts empty give O = 0, LSE = -inf."""
    rng = _rng(33)
    D = 6
    o1, o2 = _rand(rng, 3, D), _rand(rng, 3, D)
    l1 = np.array([0.3, -2.0, 5.0])
    om, lm = oracle.lse_merge(o1[None], l1[None], lib=lib)
    _close(om, o1, 0.0, "one part O")
    _close(lm, l1, 0.0, "one part LSE")
    om, lm = oracle.lse_merge(np.stack([o1, o2]), np.stack([l1, l1]), lib=lib)
    _close(om, 0.5 * (o1 + o2), 1e-15, "equal parts O")
    _close(lm, l1 + math.log(2.0), 1e-15, "equal parts LSE")
    for base in (0.0, 1000.0, -1000.0):
        lo = np.full(3, base)
        om, lm = oracle.lse_merge(np.stack([o1, o2]), np.stack([lo + math.log(3.0), lo]), lib=lib)
        # LSE near 1000 carries fp64 spacing 1.1e-13 into the weights
        _close(om, 0.75 * o1 + 0.25 * o2, 1e-12, f"3:1 parts O at {base}")
        _close(lm, lo + math.log(4.0), 1e-12, f"3:1 parts LSE at {base}")
    empty = np.full(3, -np.inf)
    om, lm = oracle.lse_merge(np.stack([o1, np.zeros_like(o2), o2 * 0]),
                              np.stack([l1, empty, empty]), lib=lib)
    _close(om, o1, 1e-15, "empty parts ignored: O")
    _close(lm, l1, 1e-15, "empty parts ignored: LSE")
    om, lm = oracle.lse_merge(np.stack([o1 * 0, o2 * 0]), np.stack([empty, empty]), lib=lib)
    assert np.all(om == 0.0) and np.all(np.isneginf(lm)), "all parts empty"


SPLIT_PINS = [pin_split_partition, pin_split_range_special_cases, pin_merge_closed_forms]


MOD_PINS = [pin_mod_window_zero, pin_mod_alibi_identical_keys, pin_mod_dense_brute_force,
            pin_mod_reduces_to_plain, pin_mod_bwd_finite_differences, pin_mod_bwd_invariants,
            pin_mod_key_padding]

FWD_PINS = [pin_hand_example, pin_identical_keys, pin_causal_row0, pin_scale_zero,
            pin_single_key, pin_library_routines, pin_softmax_rows_sum_to_one, pin_key_permutation,
            pin_gqa_equals_repeated_mha, pin_rows_match_full, pin_pages_harness,
            pin_conditional_rescale, pin_threshold_extremes]
BWD_PINS = [pin_bwd_finite_differences, pin_bwd_invariants, pin_bwd_closed_forms]
ALL_PINS = FWD_PINS + BWD_PINS + MOD_PINS + SPLIT_PINS
