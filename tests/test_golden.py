"""Golden fixtures (tests/golden/*.txt, written by tests/golden/make_golden.py from the
fp64 oracle): the oracle and the seeded input generator must keep reproducing them
(no GPU), and the CUDA path must match them in every mode (GPU)."""
import os
import sys

import numpy as np
import pytest

from helpers import GRAD_ATOL, GRAD_RTOL, LOSS_RTOL, assert_close, ensure_built

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))
import make_golden as golden  # noqa: E402


@pytest.mark.parametrize("name", sorted(golden.CASES))
def test_oracle_reproduces_golden(name):
    import oracle
    c = golden.CASES[name]
    hdr, ref = golden.read(name)
    x, y = golden.inputs(c)
    assert golden.checksum(x, y) == pytest.approx(hdr["checksum"], rel=1e-15, abs=0.0)
    loss, gx, gy = oracle.batch(x, y, c["gamma"], grad_loss=golden.weights(c))
    np.testing.assert_allclose(loss, ref["loss"], rtol=1e-12, atol=0.0)
    np.testing.assert_allclose(gx, ref["grad_x"], rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(gy, ref["grad_y"], rtol=1e-10, atol=1e-15)


@pytest.mark.gpu
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
@pytest.mark.parametrize("name", sorted(golden.CASES))
def test_cuda_matches_golden(name, mode):
    torch = pytest.importorskip("torch")
    ensure_built()
    from differentiable_series_alignment_gb300 import _lib as L
    c = golden.CASES[name]
    _, ref = golden.read(name)
    x, y = (torch.from_numpy(a).cuda() for a in golden.inputs(c))
    B, N, D = x.shape
    M = y.shape[1]
    ws = L.workspace(L.OP_FWD_BWD, B, N, M, D, mode)
    loss, gx, gy = torch.empty(B, device="cuda"), torch.empty_like(x), torch.empty_like(y)
    g = torch.from_numpy(golden.weights(c).astype(np.float32)).cuda()
    L.sdtw_forward(x, y, c["gamma"], mode, loss, ws)
    L.sdtw_backward(x, y, c["gamma"], mode, g, gx, gy, ws)
    assert L.sdtw_last_device_status(ws) == 0
    what = f"golden {name} mode={mode}"
    assert_close(loss.cpu().numpy(), ref["loss"], LOSS_RTOL, 0.0, what + " loss")
    assert_close(gx.cpu().numpy(), ref["grad_x"], GRAD_RTOL, GRAD_ATOL, what + " grad_x")
    assert_close(gy.cpu().numpy(), ref["grad_y"], GRAD_RTOL, GRAD_ATOL, what + " grad_y")
