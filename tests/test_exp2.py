"""The two exponential paths of the kernels' softmax (hardware ex2 and the cubic
on the FMA pipe) against fp64 exp2 over the range the softmax feeds them."""
import numpy as np
import pytest
import torch

import exact_attention_blackwell_tiled_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs():
    g = torch.Generator().manual_seed(0)
    # the softmax argument t - m lies in [-inf, 8] with the stale-max rescale
    dense = torch.linspace(-125.0, 8.0, 2_000_001, dtype=torch.float64)
    rnd = torch.rand(1_000_000, generator=g, dtype=torch.float64) * 133.0 - 125.0
    edges = torch.tensor([-125.0, -124.5, -1.5, -0.5, -0.25, 0.0, 0.25, 0.5, 1.5, 7.5, 8.0],
                         dtype=torch.float64)
    return torch.cat([dense, rnd, edges]).float()


@pytest.mark.parametrize("which,bound", [(0, 2.0 ** -20), (1, 1.2e-4), (2, 1.2e-4)],
                         ids=["mufu", "poly", "poly_packed"])
def test_exp2_relative_error(which, bound):
    x = _inputs()
    y = fa.exp2_test(x.cuda(), which).cpu().double().numpy()
    ref = np.exp2(x.double().numpy())
    rel = np.abs(y / ref - 1.0)
    assert rel.max() <= bound, f"max rel err {rel.max():.3e} at x={x[int(rel.argmax())].item()}"
    # well under the bf16 half-ulp the P operand is rounded to
    assert rel.max() < 2.0 ** -9


def test_exp2_poly_masked_inputs():
    x = torch.tensor([-float("inf"), -1e30, -200.0, -126.0], device="cuda")
    for which in (1, 2):
        y = fa.exp2_test(x, which).cpu()
        assert bool((y >= 0).all()) and bool((y <= 2.0 ** -124).all())
    y0 = fa.exp2_test(x, 0).cpu()
    assert bool((y0 >= 0).all()) and bool((y0 <= 2.0 ** -126).all())
    assert bool((y0[:3] == 0).all())  # below the normal range the hardware path flushes to 0
