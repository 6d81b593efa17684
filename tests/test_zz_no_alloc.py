"""sdtw_forward_noalloc, called through the C ABI: the forward for callers that
cannot allocate device memory (no allocator of their own, or no cudaMalloc
allowed in their loop) must give the losses of the workspace-based
sdtw_forward, call after call, although it reuses one static scratch array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import oracle
from differentiable_series_alignment_gb300 import synth
from helpers import LOSS_RTOL, assert_close, ensure_built

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from differentiable_series_alignment_gb300 import _lib
    return _lib


def _noalloc(lib, x, y, gamma, mode, loss):
    B, N, D = x.shape
    M = y.shape[1]
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    return lib.load().sdtw_forward_noalloc(vp(x.data_ptr()), vp(y.data_ptr()), B, N, M, D, ctypes.c_float(gamma),
                                           mode, vp(loss.data_ptr()), stream)


@pytest.mark.parametrize("mode", [0, 1])
def test_noalloc_forward_matches_workspace_forward_on_consecutive_calls(lib, mode):
    for rep, (B, N, M, D, gamma) in enumerate([(4, 64, 64, 4, 1.0), (3, 100, 37, 16, 0.5)]):
        x, y = synth.iid_normal_pair(B, N, M, D, 0, repeat=rep)
        xt, yt = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
        ref = torch.empty(B, device="cuda")
        ws = lib.workspace(lib.OP_FWD_BWD, B, N, M, D, mode)
        lib.sdtw_forward(xt, yt, gamma, mode, ref, ws)
        got = torch.full((B,), float("nan"), device="cuda")
        assert _noalloc(lib, xt, yt, gamma, mode, got) == 0
        torch.cuda.synchronize()
        assert_close(got.cpu().numpy(), ref.cpu().numpy(), LOSS_RTOL, 0.0, f"noalloc call {rep} mode {mode}")
        # and against the fp64 oracle itself (the two entries may run different forward kernels)
        ol = oracle.batch(x, y, gamma)[0]
        assert_close(got.cpu().numpy(), ol, LOSS_RTOL, 0.0, f"noalloc call {rep} mode {mode} vs oracle")


def test_noalloc_reports_a_timed_out_wait_as_nan_losses(lib):
    """A device-side wait that runs out of time (the first strip withholds its
    ready flags; no GPU fault involved) leaves NaN in the losses, and the next call
    is correct again."""
    x, y = synth.iid_normal_pair(2, 160, 40, 3, 98)
    xt, yt = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    loss = torch.zeros(2, device="cuda")
    try:
        lib.sdtw_debug_set_wait(0.05, skip_publish=True)
        assert _noalloc(lib, xt, yt, 1.0, 1, loss) == 0
        torch.cuda.synchronize()
        assert torch.isnan(loss).all()
    finally:
        lib.sdtw_debug_set_wait(0.0, skip_publish=False)
    assert _noalloc(lib, xt, yt, 1.0, 1, loss) == 0
    torch.cuda.synchronize()
    assert_close(loss.cpu().numpy(), oracle.batch(x, y, 1.0)[0], LOSS_RTOL, 0.0, "noalloc after a timeout")


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    x = torch.zeros((32, 512, 64), device="cuda")
    loss = torch.empty(32, device="cuda")
    assert _noalloc(lib, x, x, 1.0, 1, loss) == 8   # SDTW_ERR_TOO_LARGE
    # sequence lengths above 2^24 are rejected before any size arithmetic
    vp = ctypes.c_void_p
    rc = lib.load().sdtw_forward_noalloc(vp(x.data_ptr()), vp(x.data_ptr()), 1, 4, (1 << 24) + 1, 4,
                                         ctypes.c_float(1.0), 0, vp(loss.data_ptr()), None)
    assert rc == 8
