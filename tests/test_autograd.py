"""attention(): the library's forward and backward through torch.autograd."""
import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import oracle
import synth
from parity_helpers import assert_grad_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("mode", ["causal", "window_bias", "padded"])
def test_attention_autograd(mode):
    w = synth.Workload("autograd", 2, 4, 2, 300, 300, 128, mode == "causal", 40, with_do=True)
    q, k, v, do = synth.make_inputs(w, with_do=True)
    lens = torch.tensor([170, 300], dtype=torch.int32)
    if mode == "causal":
        kw = dict(causal=True)
    elif mode == "window_bias":
        kw = dict(window=(80, 20),
                  alibi_slopes=torch.tensor([0.3, -0.2, 0.1, 0.5], device="cuda"))
    else:
        kw = dict(window=(-1, 0), seqlens_k=lens.cuda())
    qd, kd, vd = (t.cuda().requires_grad_() for t in (q, k, v))
    o = fa.attention(qd, kd, vd, deterministic=True, **kw)
    o.backward(do.cuda())
    # the same bits as the direct calls
    o2, lse2 = fa.fwd(qd.detach(), kd.detach(), vd.detach(), **kw)
    g2 = fa.bwd(qd.detach(), kd.detach(), vd.detach(), o2, do.cuda(), lse2, deterministic=True,
                **kw)
    assert torch.equal(o.detach().view(torch.int16), o2.view(torch.int16))
    for a, b in zip((qd.grad, kd.grad, vd.grad), g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # and the oracle's gradients
    if mode == "causal":
        dq_r, dk_r, dv_r, _, _ = oracle.bwd(q, k, v, do, True, w.softmax_scale)
    elif mode == "padded":
        dq_r, dk_r, dv_r, _, _ = oracle.bwd_mod(q, k, v, do, w.softmax_scale, -1, 0,
                                                seqlens_k=lens)
    else:
        dq_r, dk_r, dv_r, _, _ = oracle.bwd_mod(q, k, v, do, w.softmax_scale, 80, 20,
                                                slopes=kw["alibi_slopes"].cpu())
    for g, r, n in zip((qd.grad, kd.grad, vd.grad), (dq_r, dk_r, dv_r), ("dq", "dk", "dv")):
        assert_grad_close(g, r, f"{mode} {n}")


def test_calls_from_a_thread_without_cuda_calls_of_its_own():
    """Forward and backward called from a new thread whose buffers all come from
    torch's cache, so that the thread itself has made no CUDA runtime call that
    binds the device's context (as on a framework's autograd worker thread).
    The tensor maps are built through the driver API, which needs that
    context; the results must equal the main thread's bit for bit."""
    import threading
    w = synth.Workload("thread", 1, 4, 2, 300, 300, 128, True, 7, with_do=True)
    q, k, v, do = (t.cuda() for t in synth.make_inputs(w, with_do=True))
    o, lse = fa.fwd(q, k, v, causal=True)
    ref = fa.bwd(q, k, v, o, do, lse, causal=True, deterministic=True)
    # the same sizes once more, freed, so the thread's allocations hit the cache
    tmp = fa.bwd(q, k, v, o, do, lse, causal=True, deterministic=True)
    tmp2 = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    del tmp, tmp2
    result = {}

    def run():
        try:
            o2, l2 = fa.fwd(q, k, v, causal=True)
            g2 = fa.bwd(q, k, v, o2, do, l2, causal=True, deterministic=True)
            torch.cuda.synchronize()
            result["out"] = (o2, l2, g2)
        except Exception as e:  # reported on the main thread below
            result["err"] = e

    th = threading.Thread(target=run)
    th.start()
    th.join()
    assert "err" not in result, result.get("err")
    o2, l2, g2 = result["out"]
    assert torch.equal(o2.view(torch.int16), o.view(torch.int16))
    assert torch.equal(l2, lse)
    for a, b in zip(g2, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))

