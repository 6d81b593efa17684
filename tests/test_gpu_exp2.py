"""The library's own exponential of the double-float path (exp2_neg: Cody & Waite
reduction to f in [-1/2, 1/2] and a fitted degree-7 polynomial, scaled by the
exponent bits) against the correctly rounded 2^x and against CUDA's exp2f, over
its whole range x in [-125, 0], with the bound the header states (2 ulp)."""
import numpy as np
import pytest

from helpers import ensure_built

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def ulp_distance(a, b):
    """|a - b| in units of float32 spacing, both positive finite float32 arrays."""
    ia = a.astype(np.float32).view(np.int32).astype(np.int64)
    ib = b.astype(np.float32).view(np.int32).astype(np.int64)
    return np.abs(ia - ib)


def test_exp2_neg_within_two_ulp_and_unbiased():
    ensure_built()
    from differentiable_series_alignment_gb300 import _lib as L
    g = np.random.default_rng(7)
    x = np.concatenate([g.uniform(-125.0, 0.0, 1 << 20), g.uniform(-1.0, 0.0, 1 << 18),
                        -np.arange(126, dtype=np.float64),               # integers: f = 0
                        -np.arange(126, dtype=np.float64) - 0.5,         # the ends of the reduced range
                        np.array([-125.0, -124.999, -1e-7, -0.0])]).astype(np.float32)
    x = x[x >= -125.0]
    xt = torch.from_numpy(x).cuda()
    mine = torch.empty_like(xt)
    L.sdtw_debug_exp2_neg(xt, mine)
    cuda_exp2f = torch.exp2(xt)
    torch.cuda.synchronize()
    mine, cuda_exp2f = mine.cpu().numpy(), cuda_exp2f.cpu().numpy()
    exact = np.exp2(x.astype(np.float64))
    rounded = exact.astype(np.float32)
    assert np.all(np.isfinite(mine)) and np.all(mine > 0)
    assert ulp_distance(mine, rounded).max() <= 2
    assert ulp_distance(mine, cuda_exp2f).max() <= 3
    # no systematic bias: the DP sums ~N+M of these along every path
    rel = (mine.astype(np.float64) - exact) / exact
    assert abs(rel.mean()) < 2e-9, rel.mean()


def test_exp2_neg_flushes_below_its_range():
    ensure_built()
    from differentiable_series_alignment_gb300 import _lib as L
    x = torch.tensor([-125.5, -126.0, -200.0, -1e30, float("-inf")], device="cuda")
    out = torch.full_like(x, 1.0)
    L.sdtw_debug_exp2_neg(x, out)
    assert torch.all(out == 0.0)
