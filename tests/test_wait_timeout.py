"""The kernels' bounded waits run out on the GPU without faulting it: a wait on
something that never happens returns FA_ERR_TIMEOUT through a status word, and
the CUDA context keeps working afterwards (no trap, no hang)."""
import time

import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa
import oracle
import synth
from parity_helpers import assert_fwd_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_semaphore_wait_runs_out_and_context_survives():
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")  # nothing ever sets it
    t0 = time.perf_counter()
    assert fa.wait_test(0, flag) == fa.FA_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 1.0 < elapsed < 30.0, elapsed  # the 2 s limit, not an endless spin
    flag.fill_(1)
    assert fa.wait_test(0, flag) == fa.FA_OK
    # the context still runs kernels and gives correct results
    w = synth.Workload("after_timeout", 1, 2, 2, 200, 200, 64, True, 3)
    q, k, v = synth.make_inputs(w)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK
    o_r, lse_r = oracle.fwd(q, k, v, True, w.softmax_scale)
    assert_fwd_close(o, lse, o_r, lse_r, "after a timed-out wait")


def test_mbarrier_wait_runs_out():
    assert fa.wait_test(1) == fa.FA_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert fa.fwd_status() == fa.FA_OK  # the forward's status word is untouched
