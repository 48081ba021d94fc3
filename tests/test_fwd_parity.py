"""Forward pass of the CUDA library (through the C ABI) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import oracle
import synth
from parity_helpers import (assert_fwd_close, check_guards, guarded_empty, np64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert fa.fwd_status() == fa.FA_OK, "a forward launch recorded a timed-out wait"


def _run_full(B, Hq, Hkv, Sq, Sk, D, causal, seed, scale=None, qk_std=1.0):
    w = synth.Workload("case", B, Hq, Hkv, Sq, Sk, D, causal, seed, qk_std=qk_std, scale=scale)
    q, k, v = synth.make_inputs(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, obuf = guarded_empty((B, Hq, Sq, D), torch.bfloat16, DEV)
    lse, lbuf = guarded_empty((B, Hq, Sq), torch.float32, DEV)
    fa.fwd(qd, kd, vd, causal=causal, scale=w.softmax_scale, out=o, lse=lse)
    assert fa.last_launch_count() == 1
    torch.cuda.synchronize()
    check_guards(obuf, o.numel())
    check_guards(lbuf, lse.numel())
    o_ref, lse_ref = oracle.fwd(q, k, v, causal, w.softmax_scale)
    return assert_fwd_close(o, lse, o_ref, lse_ref, f"{w}")


SMALL = [
    # B, Hq, Hkv, Sq, Sk, D, causal
    (1, 2, 2, 128, 128, 128, False),  # exactly one tile
    (1, 2, 2, 128, 128, 64, True),
    (2, 4, 2, 300, 300, 128, False),  # several tiles + ragged tail, GQA 2
    (2, 4, 2, 300, 300, 128, True),
    (1, 4, 1, 257, 257, 64, True),    # GQA 4, tail of 1 row
    (1, 2, 2, 1, 1, 128, False),      # single query, single key
    (1, 2, 2, 1, 1, 64, True),
    (1, 2, 2, 127, 129, 128, False),  # Sq != Sk
    (1, 2, 2, 129, 127, 64, True),    # causal, Sq > Sk (top-left: late rows see all keys)
    (1, 2, 1, 100, 520, 128, True),   # causal, Sk > Sq
    (1, 3, 3, 640, 384, 64, False),
    (3, 1, 1, 513, 513, 128, True),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B%dH%d-%dS%dx%dD%d%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n"))
def test_small_shapes(case):
    B, Hq, Hkv, Sq, Sk, D, causal = case
    _run_full(B, Hq, Hkv, Sq, Sk, D, causal, seed=hash(case) % 1000)


# The D = 64 forward without modifications walks each 128-key tile as two
# 64-key halves through a ring of three score buffers per query tile, and keeps
# that ring (and its barrier phases) running from one unit to the next.
RING64 = [
    (1, 2, 2, 200, 60, 64, False),     # second half of the only kv tile sees no key
    (1, 2, 2, 300, 65, 64, True),      # one key in the second half
    (1, 3, 3, 200, 192, 64, True),     # tile 1 of the pair sees one more kv tile
    (2, 40, 40, 640, 640, 64, True),   # 240 units: several per CTA, causal
    (2, 40, 8, 384, 1000, 64, False),  # 160 units, GQA 5, ragged keys
]


@pytest.mark.parametrize("case", RING64, ids=lambda c: "B%dH%d-%dS%dx%dD%d%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n"))
def test_d64_score_ring_shapes(case):
    B, Hq, Hkv, Sq, Sk, D, causal = case
    _run_full(B, Hq, Hkv, Sq, Sk, D, causal, seed=hash(case) % 1000)


def test_tiny_workload_full():
    """The tiny workload (B=1, H=2, S=256, D=64, non-causal, scale 1/8) in full."""
    w = synth.TINY
    _run_full(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.causal, w.seed, scale=w.scale)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("scale", [0.0, 1.0, 4.0])
def test_scale_extremes(scale, D):
    """scale 0 (uniform weights), and peaky softmax rows that stress the
    conditional rescale (at D = 64 the rescale waits for the previous half's
    GEMM 2 through its score buffer's barrier)."""
    _run_full(1, 2, 2, 384, 384, D, True, seed=11, scale=scale, qk_std=2.0)


def test_sq_zero_is_noop():
    q = torch.randn(1, 2, 0, 64, device=DEV).bfloat16()
    k = torch.randn(1, 2, 8, 64, device=DEV).bfloat16()
    o, lse = fa.fwd(q, k, k, causal=True)
    assert o.numel() == 0 and lse.numel() == 0
    assert fa.last_launch_count() == 0


def test_forward_is_deterministic():
    w = synth.Workload("det", 2, 4, 2, 700, 700, 128, True, 9)
    q, k, v = (t.to(DEV) for t in synth.make_inputs(w))
    o1, l1 = fa.fwd(q, k, v, causal=True)
    o2, l2 = fa.fwd(q, k, v, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _sampled(w: synth.Workload, n_per_head, full_heads):
    q, k, v = synth.make_inputs(w, with_do=False)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.fwd(qd, kd, vd, causal=w.causal, scale=w.softmax_scale)
    torch.cuda.synchronize()
    rows = synth.sample_rows(w, n_per_head=n_per_head, full_heads=full_heads)
    o_ref, lse_ref = oracle.fwd_rows(q, k, v, w.causal, w.softmax_scale, rows)
    o_g = np64(o.reshape(-1, w.D)[torch.as_tensor(rows, device=DEV)])
    l_g = np64(lse.reshape(-1)[torch.as_tensor(rows, device=DEV)])
    # properties that hold at every row: finite, O inside the hull of V's range
    assert bool(torch.isfinite(lse).all())
    assert bool(torch.isfinite(o.float()).all())
    return assert_fwd_close(o_g, l_g, o_ref, lse_ref, w.name)


def test_train_causal_sampled():
    _sampled(synth.TRAIN, 256, 2)


def test_train_noncausal_sampled():
    _sampled(synth.TRAIN_NONCAUSAL, 256, 2)


def test_gqa_spike_sampled():
    """GQA 32/8 at S=8192 with spiked keys: large late maxima exercise the
    conditional rescale."""
    _sampled(synth.GQA_SPIKE, 48, 0)


@pytest.mark.parametrize("S,D,causal", [(1024, 64, True), (4096, 128, False), (8192, 128, False),
                                        (8192, 64, False), (16384, 64, True), (32768, 128, False)])
def test_sweep_sampled(S, D, causal):
    _sampled(synth.sweep(S, D, causal), 16 if S >= 16384 else 48, 0)


def _kv_bytes(w: synth.Workload) -> int:
    return 2 * w.B * w.Hkv * w.Sk * w.D * 2


@pytest.mark.parametrize("S", [1024, 2048, 32768])
def test_sweep_causal_d128_large_kv(S):
    """Causal D=128 sweep points, whose K/V exceed L2 (128 MiB at S <= 16k,
    256 MiB at 32k): the longest-first snake deals every head's tile pairs to
    all SMs at once.  At S=32768 the 2048 units take 14 rounds of 152 CTAs with
    a partial last round.  Sampled rows of every head and two whole heads
    against the oracle."""
    w = synth.sweep(S, 128, True)
    assert _kv_bytes(w) > 64 << 20
    _sampled(w, 32, 2)


def test_bwd_workload_forward_sampled():
    """The forward of the backward workload (B=2, H=16, S=8192, D=128, causal),
    which gives the backward its O and LSE (K/V of 128 MiB).  O and LSE checked
    on sampled rows of every head and two whole heads."""
    w = synth.BWD
    assert _kv_bytes(w) > 64 << 20
    _sampled(w, 32, 2)


def test_timing_events_bracket_the_kernel():
    w = synth.Workload("t", 1, 4, 4, 1024, 1024, 128, False, 3)
    q, k, v = (t.to(DEV) for t in synth.make_inputs(w))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fa.set_timing_events(e0, e1)
    fa.fwd(q, k, v)
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0
