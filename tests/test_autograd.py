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
