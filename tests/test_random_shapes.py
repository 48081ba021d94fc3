"""Seeded random shapes through every entry point of the CUDA library against
the fp64 oracle: batch, heads, GQA group, ragged lengths, head dimension,
causal / window / bias / key padding, atomic and deterministic backward,
split-KV forward."""
import numpy as np
import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import oracle
import synth
from parity_helpers import assert_fwd_close, assert_fwd_rows, assert_grad_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 3))
    Hkv = int(rng.integers(1, 3))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    D = int(rng.choice([64, 128]))
    Sk = int(rng.integers(1, 700))
    Sq = int(rng.integers(1, 700))
    kind = rng.choice(["plain", "causal", "window", "bias"])
    wl, wr, bias = -1, -1, False
    if kind == "causal":
        wr = 0
    elif kind in ("window", "bias"):
        wr = int(rng.choice([-1, 0, int(rng.integers(0, 200))]))
        wl = int(rng.integers(max(0, Sq - Sk), max(0, Sq - Sk) + 300))
        bias = kind == "bias"
    return B, Hq, Hkv, Sq, Sk, D, wl, wr, bias


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("seed", range(16))
def test_random_shape(seed):
    B, Hq, Hkv, Sq, Sk, D, wl, wr, bias = _draw(seed)
    name = f"seed{seed} B{B} H{Hq}/{Hkv} S{Sq}x{Sk} D{D} w({wl},{wr}) bias={bias}"
    w = synth.Workload("rand", B, Hq, Hkv, Sq, Sk, D, False, 50 + seed, with_do=True)
    q, k, v, do = synth.make_inputs(w, with_do=True)
    slopes = (torch.tensor([0.3 * (-1) ** h * (1 + h % 3) for h in range(Hq)], dtype=torch.float32)
              if bias else None)
    sd = slopes.to(DEV) if slopes is not None else None
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    kw = dict(window=(wl, wr), alibi_slopes=sd)
    o, lse = fa.fwd(qd, kd, vd, scale=w.softmax_scale, **kw)
    dq_r, dk_r, dv_r, o_r, lse_r = oracle.bwd_mod(q, k, v, do, w.softmax_scale, wl, wr,
                                                  slopes=slopes)
    assert_fwd_close(o, lse, o_r, lse_r, name)
    # atomic, deterministic, and atomic with the CTA-pair kernel selected (it
    # runs where it applies: D = 128 without a window other than causal or a
    # bias; elsewhere the call takes the default kernel)
    for mode in ("atomic", "det", "pair"):
        det = mode == "det"
        ws = torch.empty(fa.bwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, det), dtype=torch.uint8,
                         device=DEV)
        prev = fa.set_bwd_kernel(fa.BWD_KERNEL_PAIR if mode == "pair" else fa.BWD_KERNEL_AUTO)
        try:
            dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, scale=w.softmax_scale, deterministic=det,
                                workspace=ws, **kw)
            assert fa.bwd_status(ws) == fa.FA_OK
        finally:
            fa.set_bwd_kernel(prev)
        tag = f"{name} {mode}"
        if wl == 0 and wr == 0:
            bound = 1e-3 * float(np.abs(dv_r).max())
            assert float(dq.float().abs().max()) <= bound, f"{tag} dQ"
            assert float(dk.float().abs().max()) <= bound, f"{tag} dK"
        else:
            assert_grad_close(dq, dq_r, f"{tag} dQ")
            assert_grad_close(dk, dk_r, f"{tag} dK")
        assert_grad_close(dv, dv_r, f"{tag} dV")
    o2, lse2 = fa.fwd(qd, kd, vd, scale=w.softmax_scale, n_splits=0, **kw)
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    assert_fwd_close(o2, lse2, o_r, lse_r, f"{name} split")


@pytest.mark.parametrize("seed", range(12))
def test_random_shape_padded(seed):
    """Per-batch key counts (0 to past Sk) with any window, rows that see no key
    included: forward, both backward modes and split-KV."""
    B, Hq, Hkv, Sq, Sk, D, _, _, bias = _draw(100 + seed)
    rng = np.random.default_rng(3000 + seed)
    B = int(rng.integers(1, 5))
    lens = rng.integers(0, Sk + 60, B).astype(np.int32)
    lens[rng.integers(0, B)] = Sk  # at least one full batch
    wl = int(rng.choice([-1, int(rng.integers(0, 400))]))
    wr = int(rng.choice([-1, 0, int(rng.integers(0, 300))]))
    name = f"seed{seed} B{B} H{Hq}/{Hkv} S{Sq}x{Sk} D{D} w({wl},{wr}) bias={bias} L={list(lens)}"
    w = synth.Workload("randpad", B, Hq, Hkv, Sq, Sk, D, False, 80 + seed, with_do=True)
    q, k, v, do = synth.make_inputs(w, with_do=True)
    slopes = (torch.tensor([0.3 * (-1) ** h * (1 + h % 3) for h in range(Hq)], dtype=torch.float32)
              if bias else None)
    lt = torch.from_numpy(lens)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    kw = dict(window=(wl, wr), alibi_slopes=None if slopes is None else slopes.to(DEV),
              seqlens_k=lt.to(DEV))
    dq_r, dk_r, dv_r, o_r, lse_r = oracle.bwd_mod(q, k, v, do, w.softmax_scale, wl, wr,
                                                  slopes=slopes, seqlens_k=lt)
    o, lse = fa.fwd(qd, kd, vd, scale=w.softmax_scale, **kw)
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    assert_fwd_rows(o, lse, o_r, lse_r, name)
    for det in (False, True):
        ws = torch.empty(fa.bwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, det), dtype=torch.uint8,
                         device=DEV)
        dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, scale=w.softmax_scale, deterministic=det,
                            workspace=ws, **kw)
        assert fa.bwd_status(ws) == fa.FA_OK
        tag = f"{name} det={det}"
        for g, r, n in ((dq, dq_r, "dQ"), (dk, dk_r, "dK"), (dv, dv_r, "dV")):
            if np.abs(r).max() == 0.0:
                assert float(g.float().abs().max()) == 0.0, f"{tag} {n} (all zero)"
            elif wl == 0 and wr == 0 and n != "dV":
                bound = 1e-3 * max(float(np.abs(dv_r).max()), 1e-30)
                assert float(g.float().abs().max()) <= bound, f"{tag} {n}"
            else:
                assert_grad_close(g, r, f"{tag} {n}")
    o2, lse2 = fa.fwd(qd, kd, vd, scale=w.softmax_scale, n_splits=0, **kw)
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    assert_fwd_rows(o2, lse2, o_r, lse_r, f"{name} split")
