"""fa_bwd_noalloc: the backward entry point for callers that cannot allocate.

Callers inside another framework's memory pool, an allocator callback or a
plugin that may only touch the buffers it is given cannot create the workspace
that fa_bwd needs.  fa_bwd_noalloc uses scratch compiled into the library
instead.  This test drives it through the C ABI, two calls in a row, and checks
its gradients against the fp64 oracle (the gradient tolerance of the other
backward tests) and against fa_bwd with its own workspace: within that
tolerance in the atomic mode, byte for byte in the deterministic mode (same
kernels, same fixed order of the dQ adds).  fa_bwd_noalloc_status reports the
status word kept in the scratch.  It lives in a file of its own so that it
runs last.
"""
import ctypes

import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import oracle
import synth
from parity_helpers import assert_grad_close, np64

pytestmark = pytest.mark.gpu

DEV = "cuda"
SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(q, k, v, o, do, lse, dq, dk, dv, w, deterministic):
    return fa.lib().fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk),
                                   _p(dv), w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, int(w.causal),
                                   float(w.softmax_scale), int(deterministic), _stream())


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
def test_noalloc_matches_oracle_and_fa_bwd_twice(deterministic, D):
    w = synth.Workload("noalloc", 2, 4, 2, 300, 300, D, True, 17, with_do=True)
    qh, kh, vh, doh = synth.make_inputs(w, with_do=True)
    q, k, v, do = (t.to(DEV) for t in (qh, kh, vh, doh))
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.softmax_scale)
    ref = fa.bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.softmax_scale,
                 deterministic=deterministic)
    torch.cuda.synchronize()
    dq_r, dk_r, dv_r, _, _ = oracle.bwd(qh, kh, vh, doh, w.causal, w.softmax_scale)
    for call in range(2):  # the scratch keeps the first call's contents
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rc = _noalloc(q, k, v, o, do, lse, dq, dk, dv, w, deterministic)
        assert rc == fa.FA_OK, fa.STATUS_NAMES.get(rc, rc)
        assert fa.lib().fa_bwd_noalloc_status(_stream()) == fa.FA_OK
        for name, got, r_or, r_fa in (("dQ", dq, dq_r, ref[0]), ("dK", dk, dk_r, ref[1]),
                                      ("dV", dv, dv_r, ref[2])):
            assert_grad_close(got, r_or, f"noalloc call {call} {name} vs oracle")
            if deterministic:
                assert torch.equal(got, r_fa), f"noalloc call {call} {name}: bits differ from fa_bwd"
            else:
                assert_grad_close(got, np64(r_fa), f"noalloc call {call} {name} vs fa_bwd")


def _rejected(w, deterministic):
    x = torch.empty(16, dtype=torch.bfloat16, device=DEV)  # never touched: rejected first
    lse = torch.empty(16, dtype=torch.float32, device=DEV)
    return _noalloc(x, x, x, x, x, lse, x, x, x, w, deterministic)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = synth.Workload("big", 4, 16, 16, 8192, 8192, 128, True, 1)
    assert fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D) > SCRATCH_BYTES
    assert _rejected(w, False) == fa.FA_ERR_WORKSPACE


def test_noalloc_deterministic_limit_is_lower():
    """32k query rows at D=128 fit the scratch with one accumulator (atomic) but
    not with the deterministic mode's four."""
    w = synth.Workload("mid", 1, 2, 2, 16384, 16384, 128, True, 1)
    assert fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, False) <= SCRATCH_BYTES
    assert fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, True) > SCRATCH_BYTES
    assert _rejected(w, True) == fa.FA_ERR_WORKSPACE
