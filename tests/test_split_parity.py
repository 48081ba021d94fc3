"""Split-KV forward (fa_fwd_split) and the log-sum-exp merge (fa_lse_merge) of
the CUDA library against the fp64 oracle."""
import numpy as np
import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import oracle
import synth
from parity_helpers import assert_fwd_close, check_guards, guarded_empty, np64

pytestmark = pytest.mark.gpu

DEV = "cuda"

# B, Hq, Hkv, Sq, Sk, D, window_left, window_right, bias, n_splits (0: automatic)
CASES = [
    (1, 2, 2, 200, 3000, 128, -1, -1, False, 0),    # short queries, long context
    (1, 2, 1, 1000, 1000, 64, -1, 0, False, 3),     # causal, GQA, ragged tail
    (1, 2, 2, 300, 2000, 128, -1, 1700, True, 4),   # bottom-right causal chunk, bias
    (1, 2, 2, 1500, 1500, 128, 100, 100, True, 5),  # rows with no key in some splits
    (2, 4, 2, 129, 1100, 64, -1, -1, False, 40),    # more splits asked than kv tiles (9)
    (1, 1, 1, 256, 256, 64, -1, 0, False, 2),       # causal, one pair, two splits
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
    return torch.tensor([0.25 * (-1) ** h * (1 + h) for h in range(Hq)], dtype=torch.float32)


def _case_id(c):
    return "B%dH%d-%dS%dx%dD%d-w%d,%d%s-n%d" % (c[:8] + ("-bias" if c[8] else "", c[9]))


@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_fwd_split(case):
    B, Hq, Hkv, Sq, Sk, D, wl, wr, bias, n = case
    w = synth.Workload("split", B, Hq, Hkv, Sq, Sk, D, False, 17)
    q, k, v = synth.make_inputs(w)
    slopes = _slopes(Hq, bias)
    sd = slopes.to(DEV) if slopes is not None else None
    o, ob = guarded_empty(q.shape, torch.bfloat16, DEV)
    lse, lb = guarded_empty((B, Hq, Sq), torch.float32, DEV)
    ws_bytes = fa.fwd_split_workspace_bytes(B, Hq, Sq, Sk, D, n)
    assert ws_bytes > 0
    ws, wb = guarded_empty((ws_bytes // 4,), torch.float32, DEV)
    fa.fwd(q.to(DEV), k.to(DEV), v.to(DEV), scale=w.softmax_scale, out=o, lse=lse,
           window=(wl, wr), alibi_slopes=sd, n_splits=n, split_workspace=ws.view(torch.uint8))
    assert fa.last_launch_count() == 2  # the split forward and the merge
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    check_guards(ob, o.numel())
    check_guards(lb, lse.numel())
    check_guards(wb, ws.numel())
    o_r, lse_r = oracle.fwd_mod(q, k, v, w.softmax_scale, wl, wr, slopes=slopes)
    assert_fwd_close(o, lse, o_r, lse_r, _case_id(case))


def test_one_split_is_the_plain_forward():
    """An effective count of 1 runs the unsplit kernel: identical bits."""
    w = synth.Workload("split1", 1, 4, 4, 4096, 4096, 128, True, 18)
    q, k, v = (t.to(DEV) for t in synth.make_inputs(w))
    o1, l1 = fa.fwd(q, k, v, causal=True)
    o2, l2 = fa.fwd(q, k, v, causal=True, n_splits=1)
    assert fa.last_launch_count() == 1
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_split_close_to_unsplit():
    """Every split count gives the unsplit result up to the merge's rounding."""
    w = synth.Workload("splitn", 1, 2, 2, 384, 2500, 128, False, 19)
    q, k, v = (t.to(DEV) for t in synth.make_inputs(w))
    o1, l1 = fa.fwd(q, k, v)
    for n in (2, 3, 7, 20):
        o2, l2 = fa.fwd(q, k, v, n_splits=n)
        assert (o1.float() - o2.float()).abs().max().item() <= 1.6e-2, n
        assert (l1 - l2).abs().max().item() <= 1e-4, n


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("n", [1, 3, 12, 25, 40])
def test_lse_merge(n, D):
    """fa_lse_merge on random parts with empty parts (-inf, O rows NaN-filled to
    show they are not read) and rows whose parts are all empty."""
    rows = 1000
    gen = torch.Generator().manual_seed(100 + n + D)
    op = torch.randn(n, rows, D, generator=gen, dtype=torch.float32)
    lp = torch.randn(n, rows, generator=gen, dtype=torch.float32) * 4.0 + 2.0
    empty = torch.rand(n, rows, generator=gen) < 0.3
    empty[:, :7] = True  # rows 0..6: every part empty
    lp[empty] = float("-inf")
    op[empty] = float("nan")
    o_r, lse_r = oracle.lse_merge(np.where(empty.numpy()[..., None], 0.0, op.double().numpy()),
                                  lp.double().numpy())
    o, ob = guarded_empty((rows, D), torch.bfloat16, DEV)
    lse, lb = guarded_empty((rows,), torch.float32, DEV)
    fa.lse_merge(op.to(DEV), lp.to(DEV), out=o, lse=lse)
    torch.cuda.synchronize()
    check_guards(ob, o.numel())
    check_guards(lb, lse.numel())
    o64, l64 = np64(o), np64(lse)
    none = empty.all(dim=0).numpy()
    assert none[:7].all()
    assert np.all(o64[none] == 0.0) and np.all(np.isneginf(l64[none])), "all-empty rows"
    assert np.all(np.isfinite(o64)) and np.all(np.isfinite(l64[~none]))
    # bf16 output: half an ulp of |O| <= 4 is 2^-7; fp32 exp / log in the weights
    assert np.abs(o64 - o_r).max() <= 1.6e-2
    assert np.abs(l64[~none] - lse_r[~none]).max() <= 1e-4


def test_split_full_size_sampled():
    """The chunked-prefill workload the split bench times (1024 queries at the end
    of a 32k context, bottom-right causal) with the automatic split count:
    sampled rows of every head against the oracle's row routine."""
    B, H, Sq, Sk, D = 1, 16, 1024, 32768, 128
    w = synth.Workload("split_prefill", B, H, H, Sq, Sk, D, False, 20)
    q, k, v = synth.make_inputs(w)
    wr = Sk - Sq
    o, lse = fa.fwd(q.to(DEV), k.to(DEV), v.to(DEV), window=(-1, wr), n_splits=0)
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    rng = np.random.default_rng(5)
    rows = np.concatenate([h * Sq + np.concatenate([[0, Sq - 1], rng.integers(0, Sq, 6)])
                           for h in range(H)])
    o_r, lse_r = oracle.fwd_rows_mod(q, k, v, w.softmax_scale, rows, -1, wr)
    assert_fwd_close(np64(o).reshape(-1, D)[rows], np64(lse).reshape(-1)[rows], o_r, lse_r,
                     "split prefill sampled")


@pytest.mark.parametrize("wr", [-1, 4999], ids=["none", "bottom_right_causal"])
def test_split_decode_rows(wr):
    """One query per head (decode) against a 5000-key context, GQA 4, the
    automatic split count."""
    B, Hq, Hkv, Sq, Sk, D = 4, 8, 2, 1, 5000, 128
    w = synth.Workload("split_decode", B, Hq, Hkv, Sq, Sk, D, False, 21)
    q, k, v = synth.make_inputs(w)
    n = fa.fwd_split_count(B, Hq, Sq, Sk)
    assert n > 1
    o, lse = fa.fwd(q.to(DEV), k.to(DEV), v.to(DEV), window=(-1, wr), n_splits=0)
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    o_r, lse_r = oracle.fwd_mod(q, k, v, w.softmax_scale, -1, wr)
    assert_fwd_close(o, lse, o_r, lse_r, f"decode n={n}")
