"""fa_bwd_noalloc: the backward entry point for callers that cannot allocate.

Callers inside another framework's memory pool, an allocator callback or a
plugin that may only touch the buffers it is given cannot create the workspace
that fa_bwd needs.  fa_bwd_noalloc uses scratch compiled into the library
instead.  This test drives it through the C ABI and checks that two calls in a
row give the same gradients as fa_bwd with its own workspace, within the
gradient tolerance the other backward tests use.  It lives in a file of its own
so that it runs last.
"""
import ctypes

import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import synth
from parity_helpers import assert_grad_close, np64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(q, k, v, o, do, lse, dq, dk, dv, w, deterministic):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fa.lib().fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk),
                                   _p(dv), w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, int(w.causal),
                                   float(w.softmax_scale), int(deterministic), stream)


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
def test_noalloc_matches_fa_bwd_twice(deterministic):
    w = synth.Workload("noalloc", 2, 4, 2, 300, 300, 128, True, 17, with_do=True)
    q, k, v, do = (t.to(DEV) for t in synth.make_inputs(w, with_do=True))
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.softmax_scale)
    ref = fa.bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.softmax_scale,
                 deterministic=deterministic)
    ref = [np64(t) for t in ref]
    for call in range(2):  # the scratch keeps the first call's contents
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rc = _noalloc(q, k, v, o, do, lse, dq, dk, dv, w, deterministic)
        assert rc == fa.FA_OK, fa.STATUS_NAMES.get(rc, rc)
        torch.cuda.synchronize()
        for name, got, r in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
            assert_grad_close(got, r, f"noalloc call {call} {name}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = synth.Workload("big", 4, 16, 16, 8192, 8192, 128, True, 1)
    need = fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D)
    assert need > (32 << 20)
    x = torch.empty(16, dtype=torch.bfloat16, device=DEV)  # never touched: rejected first
    lse = torch.empty(16, dtype=torch.float32, device=DEV)
    rc = _noalloc(x, x, x, x, x, lse, x, x, x, w, False)
    assert rc == 4, "expected FA_ERR_WORKSPACE"
