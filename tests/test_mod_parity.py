"""Score modification (sliding window, relative-position bias) of the CUDA
library, through fa_fwd_mod / fa_bwd_mod, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import oracle
import synth
from parity_helpers import assert_fwd_close, assert_grad_close, check_guards, guarded_empty

pytestmark = pytest.mark.gpu

DEV = "cuda"

# B, Hq, Hkv, Sq, Sk, D, window_left, window_right, bias
CASES = [
    (1, 2, 2, 300, 300, 64, 50, 20, True),       # window on both sides, ragged tail
    (1, 4, 2, 384, 448, 128, -1, 0, True),       # causal with bias, GQA, Sk > Sq
    (2, 2, 2, 1000, 1000, 128, 127, 0, False),   # local causal window of 128 keys
    (1, 2, 1, 700, 700, 64, -1, -1, True),       # bias alone, GQA 2
    (1, 2, 2, 256, 256, 128, 0, 0, False),       # each query sees only its own key
    (1, 2, 2, 500, 300, 128, 250, 40, True),     # Sq > Sk (window_left >= Sq - Sk)
    (1, 1, 1, 129, 700, 64, -1, 300, False),     # look-ahead limit only, Sq < Sk
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _slopes(Hq, bias):
    if not bias:
        return None
    base = [0.5, -0.25, 0.125, -1.0]
    return torch.tensor([base[h % 4] * (1 + h // 4) for h in range(Hq)], dtype=torch.float32)


def _inputs(case, seed=7):
    B, Hq, Hkv, Sq, Sk, D, wl, wr, bias = case
    w = synth.Workload("mod", B, Hq, Hkv, Sq, Sk, D, False, seed, with_do=True)
    q, k, v, do = synth.make_inputs(w, with_do=True)
    return w, q, k, v, do, _slopes(Hq, bias)


def _case_id(c):
    return "B%dH%d-%dS%dx%dD%d-w%d,%d%s" % (c[:8] + ("-bias" if c[8] else "",))


@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_fwd_mod(case):
    w, q, k, v, do, slopes = _inputs(case)
    wl, wr = case[6], case[7]
    sd = slopes.to(DEV) if slopes is not None else None
    o, ob = guarded_empty(q.shape, torch.bfloat16, DEV)
    lse, lb = guarded_empty((w.B, w.Hq, w.Sq), torch.float32, DEV)
    fa.fwd(q.to(DEV), k.to(DEV), v.to(DEV), scale=w.softmax_scale, out=o, lse=lse,
           window=(wl, wr), alibi_slopes=sd)
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    check_guards(ob, o.numel())
    check_guards(lb, lse.numel())
    o_r, lse_r = oracle.fwd_mod(q, k, v, w.softmax_scale, wl, wr, slopes=slopes)
    assert_fwd_close(o, lse, o_r, lse_r, _case_id(case))


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_bwd_mod(case, deterministic):
    w, q, k, v, do, slopes = _inputs(case)
    wl, wr = case[6], case[7]
    sd = slopes.to(DEV) if slopes is not None else None
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, scale=w.softmax_scale, window=(wl, wr), alibi_slopes=sd)
    ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, deterministic),
                     dtype=torch.uint8, device=DEV)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, scale=w.softmax_scale,
                        deterministic=deterministic, workspace=ws, window=(wl, wr),
                        alibi_slopes=sd)
    assert fa.bwd_status(ws) == fa.FA_OK
    dq_r, dk_r, dv_r, _, _ = oracle.bwd_mod(q, k, v, do, w.softmax_scale, wl, wr, slopes=slopes)
    name = _case_id(case)
    if wl == 0 and wr == 0:
        # each query sees one key: P = 1, so dS = dP - Delta = 0 and dQ = dK = 0
        # exactly; the kernel's Delta comes from the bf16-rounded O, leaving
        # rounding-level residues (bounded here against the dV scale)
        bound = 1e-3 * float(np.abs(dv_r).max())
        assert float(dq.float().abs().max()) <= bound, f"{name} dQ"
        assert float(dk.float().abs().max()) <= bound, f"{name} dK"
    else:
        assert_grad_close(dq, dq_r, f"{name} dQ")
        assert_grad_close(dk, dk_r, f"{name} dK")
    assert_grad_close(dv, dv_r, f"{name} dV")


def test_bwd_mod_deterministic_is_bit_identical():
    case = CASES[2]
    w, q, k, v, do, slopes = _inputs(case, seed=11)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, scale=w.softmax_scale, window=(case[6], case[7]))
    runs = []
    for _ in range(4):
        ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, True),
                         dtype=torch.uint8, device=DEV)
        runs.append(fa.bwd(qd, kd, vd, o, dod, lse, scale=w.softmax_scale, deterministic=True,
                           workspace=ws, window=(case[6], case[7])))
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_causal_window_matches_plain_causal():
    """window (-1, 0) without bias runs the causal kernel: identical bits."""
    w = synth.Workload("m", 1, 2, 2, 333, 333, 128, True, 5, with_do=True)
    q, k, v, do = (t.to(DEV) for t in synth.make_inputs(w, with_do=True))
    o1, l1 = fa.fwd(q, k, v, causal=True)
    o2, l2 = fa.fwd(q, k, v, window=(-1, 0))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    ws = torch.empty(fa.bwd_workspace_bytes(1, 2, 2, 333, 333, 128, True), dtype=torch.uint8,
                     device=DEV)
    g1 = fa.bwd(q, k, v, o1, do, l1, causal=True, deterministic=True, workspace=ws)
    g2 = fa.bwd(q, k, v, o2, do, l2, deterministic=True, workspace=ws, window=(-1, 0))
    for a, b in zip(g1, g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_zero_bias_matches_no_bias():
    """Slopes of zero add nothing: the bias kernel gives the plain result."""
    w = synth.Workload("m", 1, 2, 2, 260, 260, 64, False, 6)
    q, k, v = (t.to(DEV) for t in synth.make_inputs(w))
    o1, l1 = fa.fwd(q, k, v, window=(40, 10))
    o2, l2 = fa.fwd(q, k, v, window=(40, 10), alibi_slopes=torch.zeros(2, device=DEV))
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_fwd_mod_full_size_sampled():
    """A causal 1024-key window with the bias at full size (B=1, H=16, S=16384,
    D=128, the shape the bench's score-modification sweep times): sampled rows of
    every head against the oracle's row routine."""
    B, H, S, D, wl, wr = 1, 16, 16384, 128, 1023, 0
    w = synth.Workload("mod_full", B, H, H, S, S, D, False, 30)
    q, k, v = synth.make_inputs(w)
    slopes = _slopes(H, True)
    o, lse = fa.fwd(q.to(DEV), k.to(DEV), v.to(DEV), scale=w.softmax_scale, window=(wl, wr),
                    alibi_slopes=slopes.to(DEV))
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    rng = np.random.default_rng(8)
    rows = np.concatenate([h * S + np.concatenate([[0, 1023, 1024, S - 1], rng.integers(0, S, 4)])
                           for h in range(H)])
    o_r, lse_r = oracle.fwd_rows_mod(q, k, v, w.softmax_scale, rows, wl, wr, slopes=slopes)
    o64 = o.float().cpu().double().numpy().reshape(-1, D)[rows]
    l64 = lse.cpu().double().numpy().reshape(-1)[rows]
    assert_fwd_close(o64, l64, o_r, lse_r, "mod full size sampled")


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
def test_bwd_mod_sampled_units(deterministic):
    """A two-sided window with the bias, GQA 2, at S = 4096: two kv-head units
    of the backward against the fp64 backward."""
    B, Hq, Hkv, S, D, wl, wr = 1, 8, 4, 4096, 128, 700, 300
    w = synth.Workload("mod_bwd_units", B, Hq, Hkv, S, S, D, False, 31, with_do=True)
    q, k, v, do = synth.make_inputs(w, with_do=True)
    slopes = _slopes(Hq, True)
    sd = slopes.to(DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, scale=w.softmax_scale, window=(wl, wr), alibi_slopes=sd)
    ws = torch.empty(fa.bwd_workspace_bytes(B, Hq, Hkv, S, S, D, deterministic),
                     dtype=torch.uint8, device=DEV)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, scale=w.softmax_scale,
                        deterministic=deterministic, workspace=ws, window=(wl, wr),
                        alibi_slopes=sd)
    assert fa.bwd_status(ws) == fa.FA_OK
    units = [0, Hkv - 1]
    dq_r, dk_r, dv_r, _, _ = oracle.bwd_mod(q, k, v, do, w.softmax_scale, wl, wr, slopes=slopes,
                                            units=units)
    g = Hq // Hkv
    for u in units:
        hs = slice(u * g, (u + 1) * g)
        assert_grad_close(dq[0, hs], dq_r[0, hs], f"dQ unit {u}")
        assert_grad_close(dk[0, u], dk_r[0, u], f"dK unit {u}")
        assert_grad_close(dv[0, u], dv_r[0, u], f"dV unit {u}")
