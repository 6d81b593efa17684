"""Long sequences and small gamma at full size: B=8, N=M=8192, D=128, y a
time-warped copy of x plus N(0, 0.1^2) noise, gamma in {1, 0.1, 0.01}, fused
mode, plus the normalized variant. The oracle checks sampled batch elements
(each problem is independent); every output is checked to be finite."""
import numpy as np
import pytest

import oracle
from differentiable_series_alignment_gb300 import synth
from helpers import GRAD_ATOL, GRAD_RTOL, LOSS_RTOL, assert_close, ensure_built

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

B, L, D = 8, 8192, 128


@pytest.fixture(scope="module")
def data():
    ensure_built()
    return synth.warped_pair(B, L, D, 3)


@pytest.mark.parametrize("gamma,sample", [(1.0, [0, 7]), (0.1, [3]), (0.01, [5])])
def test_long_warped_fused(data, gamma, sample):
    from differentiable_series_alignment_gb300 import _lib as Lb
    x, y = data
    xt, yt = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    mode = Lb.FUSED | Lb.auto_precision(gamma, L, L)
    assert mode & Lb.EXTENDED
    ws = Lb.workspace(Lb.OP_FWD_BWD, B, L, L, D, mode)
    loss = torch.empty(B, device="cuda")
    gx, gy = torch.empty_like(xt), torch.empty_like(yt)
    g = torch.full((B,), 1.0 / B, device="cuda")
    Lb.sdtw_forward(xt, yt, gamma, mode, loss, ws)
    Lb.sdtw_backward(xt, yt, gamma, mode, g, gx, gy, ws)
    assert Lb.sdtw_last_device_status(ws) == 0
    loss, gx, gy = (t.cpu().numpy().astype(np.float64) for t in (loss, gx, gy))
    del ws
    torch.cuda.empty_cache()
    assert np.all(np.isfinite(loss)) and np.all(np.isfinite(gx)) and np.all(np.isfinite(gy))
    ol, ogx, ogy = oracle.batch(x[sample], y[sample], gamma, grad_loss=np.full(len(sample), 1.0 / B))
    assert_close(loss[sample], ol, LOSS_RTOL, 0.0, f"long gamma={gamma} loss")
    assert_close(gx[sample], ogx, GRAD_RTOL, GRAD_ATOL, f"long gamma={gamma} grad_x")
    assert_close(gy[sample], ogy, GRAD_RTOL, GRAD_ATOL, f"long gamma={gamma} grad_y")


def test_long_normalized(data):
    from differentiable_series_alignment_gb300 import _lib as Lb
    x, y = data
    gamma = 0.1
    sub = slice(0, 2)   # two pairs keep the oracle to three 8192^2 problems each
    xs, ys = np.ascontiguousarray(x[sub]), np.ascontiguousarray(y[sub])
    xt, yt = torch.from_numpy(xs).cuda(), torch.from_numpy(ys).cuda()
    nb = xs.shape[0]
    mode = Lb.FUSED | Lb.EXTENDED
    ws = Lb.workspace(Lb.OP_NORMALIZED, nb, L, L, D, mode)
    loss = torch.empty(nb, device="cuda")
    gx, gy = torch.empty_like(xt), torch.empty_like(yt)
    g = torch.full((nb,), 1.0 / nb, device="cuda")
    Lb.sdtw_normalized(xt, yt, gamma, mode, loss, g, gx, gy, ws)
    assert Lb.sdtw_last_device_status(ws) == 0
    loss, gx, gy = (t.cpu().numpy().astype(np.float64) for t in (loss, gx, gy))
    del ws
    torch.cuda.empty_cache()
    ol, ogx, ogy = oracle.normalized(xs, ys, gamma, grad_loss=np.full(nb, 1.0 / nb))
    sxx = oracle.batch(xs, xs, gamma)[0]
    syy = oracle.batch(ys, ys, gamma)[0]
    atol = 1e-4 * np.maximum(1.0, np.maximum(np.abs(sxx), np.abs(syy)))
    assert np.all(np.abs(loss - ol) <= atol + LOSS_RTOL * np.abs(ol)), (loss, ol)
    assert_close(gx, ogx, GRAD_RTOL, GRAD_ATOL, "long normalized grad_x")
    assert_close(gy, ogy, GRAD_RTOL, GRAD_ATOL, "long normalized grad_y")


def test_barycenter_full_size():
    """The barycenter workload at full size: K=64 block-wave sequences of length
    1024, D=8, gamma=1, lr=0.1, fused mode, initialised to the mean. Two steps are
    checked against the oracle from the CUDA path's own state; the remaining 98 of
    the 100 steps run on the GPU, with finite losses that end below the first."""
    from differentiable_series_alignment_gb300 import _lib as Lb
    K, T, D = 64, 1024, 8
    X = synth.block_waves(K, T, D, 4)
    mode = Lb.FUSED | Lb.auto_precision(1.0, T, T, D)
    z0 = X.astype(np.float64).mean(axis=0).astype(np.float32)
    Xt = torch.from_numpy(X).cuda()
    z = torch.from_numpy(z0.copy()).cuda()
    m, v = torch.zeros_like(z), torch.zeros_like(z)
    ws = Lb.workspace(Lb.OP_BARYCENTER, K, T, T, D, mode)
    losses = torch.empty(100, device="cuda")
    for t in (1, 2):
        zc, mc, vc = z.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
        zo, mo, vo, lref, _ = oracle.barycenter_step(zc, mc, vc, t, X, 1.0, lr=0.1)
        Lb.sdtw_barycenter_step(z, m, v, t, Xt, 1.0, 0.1, 0.9, 0.999, 1e-8, mode, losses[t - 1:t], ws)
        assert Lb.sdtw_last_device_status(ws) == 0
        assert_close(losses[t - 1:t].cpu().numpy(), [lref], LOSS_RTOL, 0.0, f"full-size barycenter step {t} loss")
        assert_close(m.cpu().numpy(), mo, GRAD_RTOL, GRAD_ATOL, f"full-size barycenter step {t} first moment")
        assert_close(z.cpu().numpy() - zc, zo - zc, 2e-3, 1e-6, f"full-size barycenter step {t} update")
    for t in range(3, 101):
        Lb.sdtw_barycenter_step(z, m, v, t, Xt, 1.0, 0.1, 0.9, 0.999, 1e-8, mode, losses[t - 1:t], ws)
    assert Lb.sdtw_last_device_status(ws) == 0
    lo = losses.cpu().numpy()
    assert np.all(np.isfinite(lo)) and np.all(np.isfinite(z.cpu().numpy()))
    assert lo[-1] < lo[0]
