"""The key padding mask (per-batch key counts, fa_score_mod.seqlens_k) and rows
that see no key, through fa_fwd_mod / fa_bwd_mod / fa_fwd_split, against the
fp64 oracle."""
import numpy as np
import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import oracle
import synth
from parity_helpers import (assert_fwd_close, assert_fwd_rows, assert_grad_close, check_guards,
                            guarded_empty, np64)

pytestmark = pytest.mark.gpu

DEV = "cuda"

# B, Hq, Hkv, Sq, Sk, D, window_left, window_right, bias, key counts (None: all)
CASES = [
    (4, 4, 2, 300, 700, 128, -1, -1, False, (700, 0, 129, 450)),  # an empty batch, 1 key past a tile
    (3, 2, 2, 500, 500, 64, -1, 0, True, (1, 256, 500)),           # causal + bias, a 1-key batch
    (2, 2, 1, 1000, 1000, 128, 100, 100, False, (333, 1000)),      # rows past 433 of batch 0 see none
    (2, 2, 2, 384, 384, 64, 20, -1, True, (128, 2000)),            # a count above Sk is Sk
    (1, 2, 2, 300, 100, 128, 50, -1, False, None),                 # window alone empties rows >= 150
    (1, 2, 2, 100, 1000, 128, -1, 20, False, None),                # kv tiles past every query
    (2, 4, 1, 200, 3000, 128, -1, -1, True, (2999, 1500)),         # long keys, GQA 4
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _case_id(c):
    lens = "all" if c[9] is None else ",".join(map(str, c[9]))
    return "B%dH%d-%dS%dx%dD%d-w%d,%d%s-L%s" % (c[:8] + ("-bias" if c[8] else "", lens))


def _inputs(case, seed=41):
    B, Hq, Hkv, Sq, Sk, D, wl, wr, bias, lens = case
    w = synth.Workload("pad", B, Hq, Hkv, Sq, Sk, D, False, seed, with_do=True)
    q, k, v, do = synth.make_inputs(w, with_do=True)
    slopes = (torch.tensor([0.3 * (-1) ** h * (1 + h % 3) for h in range(Hq)], dtype=torch.float32)
              if bias else None)
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32)
    return w, q, k, v, do, slopes, lens_t


def _dev(t):
    return None if t is None else t.to(DEV)


@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_fwd_padding(case):
    w, q, k, v, do, slopes, lens = _inputs(case)
    wl, wr = case[6], case[7]
    o, ob = guarded_empty(q.shape, torch.bfloat16, DEV)
    lse, lb = guarded_empty((w.B, w.Hq, w.Sq), torch.float32, DEV)
    fa.fwd(q.to(DEV), k.to(DEV), v.to(DEV), scale=w.softmax_scale, out=o, lse=lse,
           window=(wl, wr), alibi_slopes=_dev(slopes), seqlens_k=_dev(lens))
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    check_guards(ob, o.numel())
    check_guards(lb, lse.numel())
    o_r, lse_r = oracle.fwd_mod(q, k, v, w.softmax_scale, wl, wr, slopes=slopes, seqlens_k=lens)
    dead = assert_fwd_rows(o, lse, o_r, lse_r, _case_id(case))
    if case[9] is not None and 0 in case[9] or case[4] == 100:
        assert dead > 0  # the empty-row path ran


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_bwd_padding(case, deterministic):
    w, q, k, v, do, slopes, lens = _inputs(case)
    wl, wr = case[6], case[7]
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    kw = dict(window=(wl, wr), alibi_slopes=_dev(slopes), seqlens_k=_dev(lens))
    o, lse = fa.fwd(qd, kd, vd, scale=w.softmax_scale, **kw)
    ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, deterministic),
                     dtype=torch.uint8, device=DEV)
    ws.fill_(0xFF)  # NaN-patterned workspace: an accumulator read before written shows
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, scale=w.softmax_scale,
                        deterministic=deterministic, workspace=ws, **kw)
    assert fa.bwd_status(ws) == fa.FA_OK
    dq_r, dk_r, dv_r, _, lse_r = oracle.bwd_mod(q, k, v, do, w.softmax_scale, wl, wr,
                                                slopes=slopes, seqlens_k=lens)
    name = _case_id(case) + ("-det" if deterministic else "")
    assert_grad_close(dq, dq_r, f"{name} dQ")
    assert_grad_close(dk, dk_r, f"{name} dK")
    assert_grad_close(dv, dv_r, f"{name} dV")
    # exact zeros: dQ of rows that see no key, dK / dV of keys past the counts
    dead = np.isneginf(lse_r)
    assert np.all(np64(dq)[dead] == 0.0), f"{name}: dQ of rows with no key"
    if lens is not None:
        for b, n in enumerate(case[9]):
            n = min(n, w.Sk)
            assert float(dk[b, :, n:].abs().max() if n < w.Sk else 0) == 0.0, f"{name}: dK tail"
            assert float(dv[b, :, n:].abs().max() if n < w.Sk else 0) == 0.0, f"{name}: dV tail"


@pytest.mark.parametrize("n", [0, 3])
@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[4], CASES[6]], ids=_case_id)
def test_split_padding(case, n):
    """Split-KV with the padding mask: splits past a batch's keys are empty parts."""
    w, q, k, v, do, slopes, lens = _inputs(case)
    wl, wr = case[6], case[7]
    o, lse = fa.fwd(q.to(DEV), k.to(DEV), v.to(DEV), scale=w.softmax_scale, window=(wl, wr),
                    alibi_slopes=_dev(slopes), seqlens_k=_dev(lens), n_splits=n)
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    o_r, lse_r = oracle.fwd_mod(q, k, v, w.softmax_scale, wl, wr, slopes=slopes, seqlens_k=lens)
    assert_fwd_rows(o, lse, o_r, lse_r, _case_id(case) + f"-n{n}")


def test_padding_ignores_the_padded_keys():
    """Whatever finite values sit past the counts, every output is bit-identical."""
    case = CASES[0]
    w, q, k, v, do, slopes, lens = _inputs(case, seed=42)
    qd, dod, ld = q.to(DEV), do.to(DEV), lens.to(DEV)
    outs = []
    for fill in range(2):
        k2, v2 = k.clone(), v.clone()
        if fill:
            gen = torch.Generator().manual_seed(9)
            for b, n in enumerate(case[9]):
                k2[b, :, n:] = torch.randn(k2[b, :, n:].shape, generator=gen) * 30.0
                v2[b, :, n:] = torch.randn(v2[b, :, n:].shape, generator=gen) * 30.0
        kd, vd = k2.to(DEV), v2.to(DEV)
        o, lse = fa.fwd(qd, kd, vd, seqlens_k=ld)
        ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, True),
                         dtype=torch.uint8, device=DEV)
        g = fa.bwd(qd, kd, vd, o, dod, lse, deterministic=True, workspace=ws, seqlens_k=ld)
        outs.append((o, lse) + tuple(g))
    for a, b in zip(outs[0], outs[1]):
        if a.dtype == torch.bfloat16:
            a, b = a.float(), b.float()
        assert torch.equal(a, b)


def test_full_counts_match_no_padding():
    """Counts equal to Sk change nothing: same bits as the window kernel without
    counts."""
    w = synth.Workload("padfull", 2, 2, 2, 333, 333, 128, False, 43, with_do=True)
    q, k, v, do = (t.to(DEV) for t in synth.make_inputs(w, with_do=True))
    lens = torch.full((2,), 333, dtype=torch.int32, device=DEV)
    o1, l1 = fa.fwd(q, k, v, window=(40, 3))
    o2, l2 = fa.fwd(q, k, v, window=(40, 3), seqlens_k=lens)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    g1 = fa.bwd(q, k, v, o1, do, l1, window=(40, 3), deterministic=True)
    g2 = fa.bwd(q, k, v, o2, do, l2, window=(40, 3), deterministic=True, seqlens_k=lens)
    for a, b in zip(g1, g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_padding_full_size_sampled():
    """Causal attention over a padded batch at training size (B=4, H=16,
    S=8192, D=128; key counts from 1/4 S to S): sampled rows of every head
    against the oracle's row routine, split-KV as well."""
    B, H, S, D = 4, 16, 8192, 128
    w = synth.Workload("pad_full", B, H, H, S, S, D, False, 44)
    q, k, v = synth.make_inputs(w)
    rng = np.random.default_rng(12)
    lens = torch.tensor(rng.integers(S // 4, S + 1, B), dtype=torch.int32)
    lens[1] = S // 4 + 77
    qd, kd, vd, ld = q.to(DEV), k.to(DEV), v.to(DEV), lens.to(DEV)
    rows = np.concatenate([bh * S + np.concatenate([[0, S - 1], rng.integers(0, S, 3)])
                           for bh in range(B * H)])
    o_r, lse_r = oracle.fwd_rows_mod(q, k, v, w.softmax_scale, rows, -1, 0, seqlens_k=lens)
    for n in (None, 4):
        o, lse = fa.fwd(qd, kd, vd, window=(-1, 0), seqlens_k=ld, n_splits=n)
        torch.cuda.synchronize()
        assert fa.fwd_status() == fa.FA_OK
        assert_fwd_close(np64(o).reshape(-1, D)[rows], np64(lse).reshape(-1)[rows], o_r, lse_r,
                         f"padded full size sampled (splits {n})")


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
def test_padding_bwd_sampled_units(deterministic):
    """Backward over a padded batch (B=2, GQA 2, S=4096, a two-sided window):
    one kv-head unit of each batch against the fp64 backward."""
    B, Hq, Hkv, S, D, wl, wr = 2, 4, 2, 4096, 128, 900, 200
    w = synth.Workload("pad_bwd", B, Hq, Hkv, S, S, D, False, 45, with_do=True)
    q, k, v, do = synth.make_inputs(w, with_do=True)
    lens = torch.tensor([1717, 4000], dtype=torch.int32)
    qd, kd, vd, dod, ld = (t.to(DEV) for t in (q, k, v, do, lens))
    o, lse = fa.fwd(qd, kd, vd, window=(wl, wr), seqlens_k=ld)
    ws = torch.empty(fa.bwd_workspace_bytes(B, Hq, Hkv, S, S, D, deterministic),
                     dtype=torch.uint8, device=DEV)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, deterministic=deterministic, workspace=ws,
                        window=(wl, wr), seqlens_k=ld)
    assert fa.bwd_status(ws) == fa.FA_OK
    units = [0, 1 * Hkv + 1]
    dq_r, dk_r, dv_r, _, _ = oracle.bwd_mod(q, k, v, do, w.softmax_scale, wl, wr, units=units,
                                            seqlens_k=lens)
    g = Hq // Hkv
    for u in units:
        b, hk = divmod(u, Hkv)
        hs = slice(hk * g, (hk + 1) * g)
        assert_grad_close(dq[b, hs], dq_r[b, hs], f"dQ unit {u}")
        assert_grad_close(dk[b, hk], dk_r[b, hk], f"dK unit {u}")
        assert_grad_close(dv[b, hk], dv_r[b, hk], f"dV unit {u}")
