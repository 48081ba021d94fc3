"""Backward pass of the CUDA library (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import oracle
import synth
from parity_helpers import assert_grad_close, check_guards, guarded_empty, np64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _bwd_case(w: synth.Workload, deterministic: bool, units=None, guards=False):
    q, k, v, do = synth.make_inputs(w, with_do=True)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=w.causal, scale=w.softmax_scale)
    need = fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, deterministic)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    if guards:
        dq, bq = guarded_empty(q.shape, torch.bfloat16, DEV)
        dk, bk = guarded_empty(k.shape, torch.bfloat16, DEV)
        dv, bv = guarded_empty(v.shape, torch.bfloat16, DEV)
    else:
        dq = dk = dv = None
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, causal=w.causal, scale=w.softmax_scale,
                        deterministic=deterministic, workspace=ws, dq=dq, dk=dk, dv=dv)
    assert fa.bwd_status(ws) == fa.FA_OK, "backward recorded a timed-out wait"
    if guards:
        for t, b in ((dq, bq), (dk, bk), (dv, bv)):
            check_guards(b, t.numel())
    dq_r, dk_r, dv_r, _, _ = oracle.bwd(q, k, v, do, w.causal, w.softmax_scale, units=units)
    return (dq, dk, dv), (dq_r, dk_r, dv_r), (qd, kd, vd, o, dod, lse, ws)


def _compare(got, ref, w, units=None):
    dq, dk, dv = got
    dq_r, dk_r, dv_r = ref
    if units is None:
        assert_grad_close(dq, dq_r, f"{w.name} dQ")
        assert_grad_close(dk, dk_r, f"{w.name} dK")
        assert_grad_close(dv, dv_r, f"{w.name} dV")
        return
    g = w.Hq // w.Hkv
    for u in units:
        b, hk = divmod(int(u), w.Hkv)
        hs = slice(hk * g, (hk + 1) * g)
        assert_grad_close(dq[b, hs], dq_r[b, hs], f"{w.name} dQ unit {u}")
        assert_grad_close(dk[b, hk], dk_r[b, hk], f"{w.name} dK unit {u}")
        assert_grad_close(dv[b, hk], dv_r[b, hk], f"{w.name} dV unit {u}")


SMALL = [
    # B, Hq, Hkv, Sq, Sk, D, causal
    (1, 1, 1, 128, 128, 128, False),
    (1, 2, 2, 128, 128, 64, True),
    (2, 4, 2, 300, 300, 128, True),   # ragged tail, GQA 2
    (2, 4, 2, 300, 300, 128, False),
    (1, 4, 1, 257, 257, 64, False),   # GQA 4
    (1, 2, 2, 1, 1, 128, True),
    (1, 2, 2, 127, 200, 64, True),    # Sk > Sq: keys past the last query get zero grads
    (1, 2, 2, 200, 127, 128, True),   # Sq > Sk
    (1, 2, 1, 390, 260, 128, False),
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B%dH%d-%dS%dx%dD%d%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n"))
def test_small_shapes(case, deterministic):
    B, Hq, Hkv, Sq, Sk, D, causal = case
    w = synth.Workload("bwd_small", B, Hq, Hkv, Sq, Sk, D, causal, 21 + Sq, with_do=True)
    got, ref, _ = _bwd_case(w, deterministic, guards=True)
    _compare(got, ref, w)


def test_deterministic_is_bit_identical():
    w = synth.Workload("det", 2, 4, 2, 700, 700, 128, True, 5, with_do=True)
    got, ref, (qd, kd, vd, o, dod, lse, ws) = _bwd_case(w, True)
    _compare(got, ref, w)
    for _ in range(4):
        again = fa.bwd(qd, kd, vd, o, dod, lse, causal=True, scale=w.softmax_scale,
                       deterministic=True, workspace=ws)
        for a, b in zip(got, again):
            assert torch.equal(a, b), "deterministic backward differs between runs"


DET_WORKLOADS = [
    # causal calls are dealt longest first in a snake over all heads, each
    # block's chain ascending over the kv tiles: the training-scale step and
    # the backward workload (q and dO of 64 and 128 MiB)
    (synth.TRAIN.with_(with_do=True), True),
    (synth.BWD, True),
    # non-causal: head-major dealing, chains descending
    (synth.BWD.with_(name="bwd_noncausal", causal=False), False),
    # D = 64 runs the 64-row kernel, where a drain warp without head-dim rows
    # raises the semaphores: causal (units from the global counter) and
    # non-causal (static head-major dealing)
    (synth.BWD.with_(name="bwd_d64", D=64), True),
    (synth.BWD.with_(name="bwd_d64_noncausal", D=64, causal=False), False),
]


@pytest.mark.parametrize("w,snake", DET_WORKLOADS, ids=lambda x: getattr(x, "name", ""))
def test_deterministic_bit_identical_at_workload_size(w, snake):
    """The deterministic backward gives the same bits on five runs at full
    workload size, on both chain orders."""
    assert w.causal == snake, "dealing order changed"
    q, k, v, do = (t.to(DEV) for t in synth.make_inputs(w, with_do=True))
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.softmax_scale)
    ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, True),
                     dtype=torch.uint8, device=DEV)
    first = fa.bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.softmax_scale,
                   deterministic=True, workspace=ws)
    first = [t.clone() for t in first]
    assert fa.bwd_status(ws) == fa.FA_OK
    for run in range(4):
        again = fa.bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.softmax_scale,
                       deterministic=True, workspace=ws)
        assert fa.bwd_status(ws) == fa.FA_OK
        for name, a, b in zip(("dQ", "dK", "dV"), first, again):
            assert torch.equal(a, b), f"{w.name}: deterministic {name} differs on run {run + 2}"


def test_bwd_workload_sampled_heads():
    """The backward workload (B=2, H=16, S=8192, D=128, causal) at full size;
    two kv heads are checked against the full fp64 backward, every output is
    checked for finiteness, and both dQ accumulation modes agree."""
    w = synth.BWD
    units = [3, 2 * w.Hkv - 1]
    got, ref, args = _bwd_case(w, False, units=units)
    _compare(got, ref, w, units)
    for t in got:
        assert bool(torch.isfinite(t.float()).all())
    qd, kd, vd, o, dod, lse, _ = args
    det = fa.bwd(qd, kd, vd, o, dod, lse, causal=True, scale=w.softmax_scale, deterministic=True)
    _compare(det, ref, w, units)


def test_bwd_head_groups_partial_last_group():
    """Causal D=128 with atomic dQ deals its units from a counter over groups
    of kv heads sized to L2: here 21 kv heads (B=3, Hkv=7, GQA 2, S=4096) in
    groups of 9, 9 and 3.  kv heads at the group boundaries against the fp64
    backward, every output finite; then the deterministic mode on the same
    shape."""
    w = synth.Workload("head_groups", 3, 14, 7, 4096, 4096, 128, True, 12, with_do=True)
    units = [0, 8, 9, 20]
    got, ref, args = _bwd_case(w, False, units=units)
    _compare(got, ref, w, units)
    for t in got:
        assert bool(torch.isfinite(t.float()).all())
    # the deterministic mode on the same GQA shape: units from the counter over
    # all 21 kv heads, two query heads per unit behind the semaphore chain;
    # against the fp64 backward and bit-identical on a second run
    qd, kd, vd, o, dod, lse, _ = args
    det = fa.bwd(qd, kd, vd, o, dod, lse, causal=True, scale=w.softmax_scale, deterministic=True)
    _compare(det, ref, w, units)
    again = fa.bwd(qd, kd, vd, o, dod, lse, causal=True, scale=w.softmax_scale, deterministic=True)
    for a, b in zip(det, again):
        assert torch.equal(a, b), "deterministic backward differs between runs"


@pytest.fixture
def pair_kernel():
    prev = fa.set_bwd_kernel(fa.BWD_KERNEL_PAIR)
    yield
    fa.set_bwd_kernel(prev)


PAIR_SHAPES = [c for c in SMALL if c[5] == 128] + [
    (1, 2, 2, 640, 640, 128, True),    # 5 kv tiles: the last pair's second tile holds no key
    (2, 4, 1, 512, 900, 128, False),   # GQA 4, ragged Sk (8 tiles, the last partial)
    (1, 1, 1, 1000, 1000, 128, True),  # ragged Sq and Sk, causal union of the pair's blocks
]


@pytest.mark.parametrize("case", PAIR_SHAPES, ids=lambda c: "B%dH%d-%dS%dx%dD%d%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n"))
def test_pair_kernel_small_shapes(case, pair_kernel):
    """The CTA-pair main kernel (2-CTA MMA, dQ reduced over 256 keys before the
    global adds) against the fp64 backward."""
    B, Hq, Hkv, Sq, Sk, D, causal = case
    w = synth.Workload("bwd_pair", B, Hq, Hkv, Sq, Sk, D, causal, 31 + Sq, with_do=True)
    got, ref, _ = _bwd_case(w, False, guards=True)
    _compare(got, ref, w)


def test_pair_kernel_bwd_workload_sampled_heads(pair_kernel):
    """The CTA-pair kernel at the backward workload's full size (B=2, H=16,
    S=8192, causal): two kv heads against the fp64 backward, all outputs finite."""
    w = synth.BWD
    units = [3, 2 * w.Hkv - 1]
    got, ref, _ = _bwd_case(w, False, units=units)
    _compare(got, ref, w, units)
    for t in got:
        assert bool(torch.isfinite(t.float()).all())


def test_sq_zero_gives_zero_key_grads():
    k = torch.randn(1, 2, 200, 128, device=DEV).bfloat16()
    v = torch.randn(1, 2, 200, 128, device=DEV).bfloat16()
    q = torch.empty(1, 2, 0, 128, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(1, 2, 0, device=DEV)
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    _, dk, dv = fa.bwd(q, k, v, q, q, lse, causal=True, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert bool((dk == 0).all()) and bool((dv == 0).all())


def test_pair_kernel_sq_zero_gives_zero_key_grads(pair_kernel):
    """With no queries every pair unit has no block: the pair kernel still loads
    K / V and writes dK = dV = 0, including an odd kv-tile count (3 tiles)."""
    k = torch.randn(1, 2, 300, 128, device=DEV).bfloat16()
    v = torch.randn(1, 2, 300, 128, device=DEV).bfloat16()
    q = torch.empty(1, 2, 0, 128, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(1, 2, 0, device=DEV)
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    _, dk, dv = fa.bwd(q, k, v, q, q, lse, causal=True, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert bool((dk == 0).all()) and bool((dv == 0).all())


def test_timeout_status_is_clear_after_normal_runs():
    w = synth.Workload("st", 1, 2, 2, 256, 256, 64, True, 1, with_do=True)
    got, ref, (qd, kd, vd, o, dod, lse, ws) = _bwd_case(w, False)
    assert fa.bwd_status(ws) == fa.FA_OK
