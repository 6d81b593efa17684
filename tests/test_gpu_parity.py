"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Tolerances: losses rel 1e-4; gradients rel 1e-3 with abs 1e-5, the upstream
gradient being the 1/B of a batch mean. The CUDA library must be the code that
runs: every call goes through libsdtw.so.
"""
import numpy as np
import pytest

import oracle
from differentiable_series_alignment_gb300 import synth
from helpers import GRAD_ATOL, GRAD_RTOL, LOSS_RTOL, assert_close, ensure_built

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _lib():
    from differentiable_series_alignment_gb300 import _lib
    return _lib


class options:
    """Force kernel choices of the library for the duration of a block (its testing
    hook sdtw_debug_set_options): warps per wavefront CTA, which sets the strip
    count, and the difference-form cost kernels in place of the tensor-core ones."""

    def __init__(self, warps_fwd=0, warps_bwd=None, simt=False):
        self.kw = dict(warps_fwd=warps_fwd, warps_bwd=warps_fwd if warps_bwd is None else warps_bwd,
                       dist_simt=simt, fused_simt=simt)

    def __enter__(self):
        _lib().sdtw_debug_set_options(**self.kw)

    def __exit__(self, *a):
        _lib().sdtw_debug_set_options()


def warps(fwd, bwd=None):
    return options(warps_fwd=fwd, warps_bwd=bwd)


class clusters:
    """Cap the CTAs per wavefront cluster for the duration of a block (the testing
    hook sdtw_debug_set_clusters; 1: no clusters)."""

    def __init__(self, c):
        self.c = c

    def __enter__(self):
        _lib().sdtw_debug_set_clusters(self.c)

    def __exit__(self, *a):
        _lib().sdtw_debug_set_clusters(0)


def run_cuda(x, y, gamma, mode, grad_loss=None, want_grads=True):
    L = _lib()
    xt = torch.from_numpy(x).cuda()
    yt = torch.from_numpy(y).cuda()
    B, N, D = x.shape
    M = y.shape[1]
    ws = L.workspace(L.OP_FWD_BWD, B, N, M, D, mode)
    loss = torch.empty(B, device="cuda")
    L.sdtw_forward(xt, yt, gamma, mode, loss, ws)
    out = dict(loss=loss)
    if want_grads:
        g = torch.full((B,), 1.0 / B, device="cuda") if grad_loss is None else torch.from_numpy(
            np.asarray(grad_loss, np.float32)).cuda()
        gx = torch.empty_like(xt)
        gy = torch.empty_like(yt)
        L.sdtw_backward(xt, yt, gamma, mode, g, gx, gy, ws)
        out.update(gx=gx, gy=gy)
    assert L.sdtw_last_device_status(ws) == 0
    torch.cuda.synchronize()
    return {k: v.cpu().numpy().astype(np.float64) for k, v in out.items()}


def check_against_oracle(x, y, gamma, mode, grad_loss=None, sample=None, what=""):
    got = run_cuda(x, y, gamma, mode, grad_loss)
    B = x.shape[0]
    gl = np.full(B, 1.0 / B) if grad_loss is None else np.asarray(grad_loss, np.float64)
    idx = np.arange(B) if sample is None else np.asarray(sample)
    ol, ogx, ogy = oracle.batch(x[idx], y[idx], gamma, grad_loss=gl[idx])
    assert_close(got["loss"][idx], ol, LOSS_RTOL, 0.0, f"{what} loss")
    assert_close(got["gx"][idx], ogx, GRAD_RTOL, GRAD_ATOL, f"{what} grad_x")
    assert_close(got["gy"][idx], ogy, GRAD_RTOL, GRAD_ATOL, f"{what} grad_y")
    return got


MODES = [("unfused", 0), ("fused", 1)]

# Upstream gradients. The fp32 modes are checked at each test's own batch mean:
# per-pair weights of magnitude 1/B for the test's batch of B, alternating in
# sign so that a mix-up of problems shows. Their state is single precision, so
# the absolute gradient error grows with the weight; where a small batch's mean
# is beyond what the fp32 state holds at a shape (D > 4: auto_precision keeps
# fp32 only for batches of B >= 32), the test's batch is B = 32, the size of the
# configs' batches. The double-float mode is checked with O(1) weights (WEIGHTS_O1).
WEIGHTS_O1 = [0.5, -1.25, 2.0]


def mean_weights(B, signed=True):
    """Per-pair upstream weights of a batch-mean loss over B pairs (signs alternate when `signed`)."""
    return [((-1.0) ** b if signed else 1.0) / B for b in range(B)]


# --------------------------------------------------------------------------- small config

@pytest.mark.parametrize("mname,mode", MODES)
def test_small_config(mname, mode):
    c = synth.WORKLOADS["small"]
    x, y = synth.iid_normal_pair(c["B"], c["N"], c["M"], c["D"], c["seed"])
    check_against_oracle(x, y, 1.0, mode, what=f"small {mname}")


@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("N,M,D", [(1, 1, 3), (1, 7, 2), (9, 1, 1), (2, 2, 5), (31, 33, 3), (33, 31, 4),
                                   (64, 65, 7), (100, 37, 16), (37, 100, 1), (129, 130, 9)])
def test_ragged_shapes(mname, mode, N, M, D):
    x, y = synth.iid_normal_pair(3, N, M, D, 90, repeat=N * 1000 + M)
    check_against_oracle(x, y, 0.7, mode, grad_loss=mean_weights(3), what=f"{N}x{M}x{D} {mname}")


# Wide features in fp32. D=127 is the widest operand the gradient contraction
# stacks as [hi; lo] in one MMA (N = 256); the loss is the batch mean (upstream
# gradient 1/B), the setting the tolerance is stated for. (D=128 and D=256, the
# three-product path, run in the sweep above.)
@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("N,M,D", [(130, 257, 127)])
def test_wide_features_fp32(mname, mode, N, M, D):
    x, y = synth.iid_normal_pair(3, N, M, D, 90, repeat=N * 1000 + M)
    check_against_oracle(x, y, 1.0, mode, what=f"{N}x{M}x{D} {mname}")


# With O(1) per-problem upstream gradients and gamma < 1, fp32 costs and DP state
# miss abs 1e-5 on near-zero gradient entries at these widths; auto_precision
# selects the extended mode, which must then hold the tolerance. D=400 is the
# largest feature width the library accepts.
@pytest.mark.parametrize("mname,base", MODES)
@pytest.mark.parametrize("N,M,D", [(130, 257, 127), (200, 70, 128), (300, 333, 400)])
def test_wide_features_auto_precision(mname, base, N, M, D):
    L = _lib()
    mode = base | L.auto_precision(0.7, N, M, D)
    assert mode & L.EXTENDED
    x, y = synth.iid_normal_pair(3, N, M, D, 90, repeat=N * 1000 + M)
    check_against_oracle(x, y, 0.7, mode, grad_loss=WEIGHTS_O1, what=f"{N}x{M}x{D} auto {mname}")


@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("W", [1, 2, 3, 16])
def test_strip_decompositions_agree(mname, mode, W):
    # Many strips (W=1: every 32-row block its own CTA, boundaries through global
    # memory) down to one strip per problem; all must reproduce the oracle.
    x, y = synth.iid_normal_pair(2, 200, 150, 6, 91)
    with warps(W):
        check_against_oracle(x, y, 1.0, mode, what=f"W={W} {mname}")


@pytest.mark.parametrize("gamma", [10.0, 1.0, 0.1, 0.01, 0.001])
def test_small_gamma_no_nan(gamma):
    # precision chosen as the high-level API does (double-float state below gamma 0.05)
    L = _lib()
    mode = L.FUSED | L.auto_precision(gamma, 300, 300)
    x, y = synth.warped_pair(2, 300, 8, 93)
    got = check_against_oracle(x, y, gamma, mode, what=f"gamma={gamma}")
    assert all(np.all(np.isfinite(v)) for v in got.values())


@pytest.mark.parametrize("mname,mode", [("unfused+extended", 2), ("fused+extended", 3)])
@pytest.mark.parametrize("N,M,D", [(1, 1, 3), (1, 7, 2), (9, 1, 1), (31, 33, 3), (100, 37, 16), (129, 130, 9)])
def test_extended_precision_shapes(mname, mode, N, M, D):
    x, y = synth.iid_normal_pair(3, N, M, D, 92, repeat=N * 1000 + M)
    check_against_oracle(x, y, 0.7, mode, grad_loss=WEIGHTS_O1, what=f"{N}x{M}x{D} {mname}")


# The extended modes take their double-float costs from exact tensor-core level
# sums (fixed-point digits, integer level sums), in both modes up to D = 400: five
# 8-bit digits up to D = 128, six 7-bit digits above. The difference-form kernels
# (the debug option) compute the same costs on the FP32 pipe. Both must hold the tolerance at O(1) weights and agree closely. The shapes
# run the tensor-memory rings round several times (M up to 520 columns), over
# several 128-row strips, and through one, two and several K-blocks.
XTC_SHAPES = [(1, 9, 3), (33, 31, 1), (100, 37, 16), (129, 130, 63), (70, 91, 64), (130, 97, 65),
              (200, 150, 128), (300, 333, 128), (257, 520, 96), (129, 70, 129)]
XTC_WIDE = [(64, 33, 256), (300, 333, 400), (131, 77, 200), (260, 300, 256)]


@pytest.mark.parametrize("mname,mode,N,M,D", [("fused+extended", 3) + s for s in XTC_SHAPES + XTC_WIDE] +
                         [("unfused+extended", 2) + s for s in XTC_SHAPES + XTC_WIDE])
def test_extended_tensor_core_costs(mname, mode, N, M, D):
    x, y = synth.iid_normal_pair(3, N, M, D, 106, repeat=N * 1000 + D)
    got = check_against_oracle(x, y, 0.7, mode, grad_loss=WEIGHTS_O1, what=f"{mname} tc {N}x{M}x{D}")
    with options(simt=True):
        ref = run_cuda(x, y, 0.7, mode, grad_loss=WEIGHTS_O1)
    assert_close(got["loss"], ref["loss"], 1e-6, 0.0, f"{mname} tc vs difference form {N}x{M}x{D} loss")
    assert_close(got["gx"], ref["gx"], 1e-4, 1e-7, f"{mname} tc vs difference form {N}x{M}x{D} grad_x")


@pytest.mark.parametrize("W", [1, 3])
def test_extended_strip_decompositions(W):
    x, y = synth.iid_normal_pair(2, 200, 150, 6, 91)
    with warps(W):
        check_against_oracle(x, y, 0.05, 3, what=f"extended W={W}")


# Strips of 9 to 12 warps take the double-float backward's 384-thread build (wider
# requests are capped at 12 warps); both modes, 13 row blocks per problem.
@pytest.mark.parametrize("mname,mode", [("unfused+extended", 2), ("fused+extended", 3)])
@pytest.mark.parametrize("W", [10, 16])
def test_extended_wide_backward_strips(mname, mode, W):
    x, y = synth.iid_normal_pair(2, 410, 150, 6, 108)
    with warps(W):
        check_against_oracle(x, y, 0.3, mode, grad_loss=[0.5, -1.25], what=f"{mname} W={W}")


# In the fused fp32 forward with tensor-core costs, consecutive 128-row strips of a
# problem that share a thread-block cluster pass their boundary rows through each
# other's shared memory; the others through global memory. The arithmetic is the
# same either way: clusters of 4, of 2 and none give identical bits, and match the
# oracle. Strip counts 5, 3, 2 and 4 (N = 520, 300, 200, 512): the last cluster of
# a problem can be ragged (CTAs past the last strip); N = 129 has a partial strip.
@pytest.mark.parametrize("B,N,M,D", [(3, 300, 257, 3), (3, 520, 130, 3), (3, 129, 100, 2), (3, 200, 64, 3),
                                     (32, 512, 512, 64)])
def test_cluster_handoff_is_bit_identical(B, N, M, D):
    x, y = synth.iid_normal_pair(B, N, M, D, 91, repeat=N * 1000 + M)
    w = mean_weights(B)
    mname, mode, W = "fused", 1, 0
    outs = {}
    for c in (1, 2, 4):
        with clusters(c):
            outs[c] = run_cuda(x, y, 0.9, mode, grad_loss=w)
    for c in (2, 4):
        for k in outs[1]:
            np.testing.assert_array_equal(outs[c][k], outs[1][k], err_msg=f"{mname} clusters<={c} {k}")
    idx = np.arange(min(B, 3))
    ol, ogx, ogy = oracle.batch(x[idx], y[idx], 0.9, grad_loss=np.asarray(w, np.float64)[idx])
    what = f"{N}x{M}x{D} W={W} {mname}"
    assert_close(outs[4]["loss"][idx], ol, LOSS_RTOL, 0.0, f"{what} loss")
    assert_close(outs[4]["gx"][idx], ogx, GRAD_RTOL, GRAD_ATOL, f"{what} grad_x")
    assert_close(outs[4]["gy"][idx], ogy, GRAD_RTOL, GRAD_ATOL, f"{what} grad_y")


def test_fused_equals_unfused():
    # Both cost kernels exist in both modes: the tensor-core norm form (default,
    # D <= 64) and the difference form (selected through sdtw_debug_set_options). With the
    # same cost kernel the fused forward recomputes exactly the costs the unfused
    # mode stores, so the two modes agree to rounding; across cost kernels they
    # agree to the parity tolerance.
    x, y = synth.iid_normal_pair(4, 96, 80, 12, 94)
    tc_u = run_cuda(x, y, 1.0, 0)
    tc_f = run_cuda(x, y, 1.0, 1)
    with options(simt=True):
        df_u = run_cuda(x, y, 1.0, 0)
        df_f = run_cuda(x, y, 1.0, 1)
    for what, a, b in (("tensor-core costs", tc_u, tc_f), ("difference-form costs", df_u, df_f)):
        assert_close(b["loss"], a["loss"], 1e-5, 0.0, f"fused vs unfused ({what}) loss")
        assert_close(b["gx"], a["gx"], 1e-4, 1e-6, f"fused vs unfused ({what}) grad_x")
        assert_close(b["gy"], a["gy"], 1e-4, 1e-6, f"fused vs unfused ({what}) grad_y")
    assert_close(tc_f["loss"], df_f["loss"], LOSS_RTOL, 0.0, "tensor-core vs difference-form costs, loss")
    assert_close(tc_f["gx"], df_f["gx"], GRAD_RTOL, GRAD_ATOL, "tensor-core vs difference-form costs, grad_x")


@pytest.mark.parametrize("mname,mode", MODES)
def test_difference_form_cost_kernels(mname, mode):
    # the difference-form cost path at a width the tensor cores would otherwise
    # handle; a batch of 32 at its own mean (D = 20 > 4)
    x, y = synth.iid_normal_pair(32, 70, 91, 20, 96)
    with options(simt=True):
        check_against_oracle(x, y, 0.8, mode, grad_loss=mean_weights(32), what=f"difference-form {mname}")


# Wide features in fp32: beyond one K-block (D > 64) the costs come from the exact
# difference-form kernels; batches of 32 at their own mean. Ragged shapes.
@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("N,M,D", [(130, 97, 96), (200, 150, 128)])
def test_wide_features_fp32_batch_mean(mname, mode, N, M, D):
    x, y = synth.iid_normal_pair(32, N, M, D, 104, repeat=N * 1000 + D)
    check_against_oracle(x, y, 1.0, mode, grad_loss=mean_weights(32), what=f"wide {N}x{M}x{D} {mname}")


def test_distance_kernel_matches_definition():
    L = _lib()
    x, y = synth.iid_normal_pair(3, 70, 45, 9, 95)
    C = torch.empty((3, 70, 45), device="cuda")
    L.sdtw_distance(torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda(), C)
    x64, y64 = x.astype(np.float64), y.astype(np.float64)
    ref = ((x64[:, :, None, :] - y64[:, None, :, :]) ** 2).sum(-1)
    assert_close(C.cpu().numpy(), ref, 1e-5, 1e-5, "distance")


# --------------------------------------------------------------------------- headline config

@pytest.mark.parametrize("mname,mode", MODES)
def test_headline_config(mname, mode):
    c = synth.WORKLOADS["headline"]
    x, y = synth.iid_normal_pair(c["B"], c["N"], c["M"], c["D"], c["seed"])
    check_against_oracle(x, y, 1.0, mode, what=f"headline {mname}")


# --------------------------------------------------------------------------- sweep (sampled)

# Every point of the Figure 1 sweep (B=32; L at D=128, D at L=256), the whole batch,
# in the precision the high-level API picks for it (double-float above D = 64).
SWEEP_POINTS = [(128, 128), (256, 128), (512, 128), (1024, 128), (2048, 128),
                (256, 1), (256, 4), (256, 16), (256, 64), (256, 256)]


@pytest.mark.parametrize("mname,base", MODES)
@pytest.mark.parametrize("L,D", SWEEP_POINTS)
def test_sweep(mname, base, L, D):
    mode = base | _lib().auto_precision(1.0, L, L, D, 32)
    x, y = synth.iid_normal_pair(32, L, L, D, 2, repeat=L * 1000 + D)
    check_against_oracle(x, y, 1.0, mode, what=f"sweep L={L} D={D} {mname} mode={mode}")


# The fp32 modes at the sweep's wide points (difference-form costs), sampled problems.
@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("L,D", [(256, 128), (2048, 128), (256, 256)])
def test_sweep_fp32_wide_sampled(mname, mode, L, D):
    x, y = synth.iid_normal_pair(32, L, L, D, 2, repeat=L * 1000 + D)
    check_against_oracle(x, y, 1.0, mode, sample=[0, 7, 31], what=f"sweep fp32 L={L} D={D} {mname}")


# --------------------------------------------------------------------------- normalized

def run_normalized(x, y, gamma, mode, grad_loss):
    L = _lib()
    xt, yt = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    B, N, D = x.shape
    ws = L.workspace(L.OP_NORMALIZED, B, N, N, D, mode)
    loss = torch.empty(B, device="cuda")
    gx, gy = torch.empty_like(xt), torch.empty_like(yt)
    g = torch.from_numpy(np.asarray(grad_loss, np.float32)).cuda()
    L.sdtw_normalized(xt, yt, gamma, mode, loss, g, gx, gy, ws)
    assert L.sdtw_last_device_status(ws) == 0
    return loss.cpu().numpy(), gx.cpu().numpy(), gy.cpu().numpy()


@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("N,D", [(64, 4), (77, 3)])
def test_normalized(mname, mode, N, D):
    x, y = synth.iid_normal_pair(4, N, N, D, 96)
    gl = np.array([0.25, 0.25, -0.5, 1.0])
    loss, gx, gy = run_normalized(x, y, 0.8, mode, gl)
    ol, ogx, ogy = oracle.normalized(x, y, 0.8, grad_loss=gl)
    sxx = oracle.batch(x, x, 0.8)[0]
    syy = oracle.batch(y, y, 0.8)[0]
    atol = 1e-4 * np.maximum(1.0, np.maximum(np.abs(sxx), np.abs(syy)))
    assert np.all(np.abs(loss - ol) <= atol + LOSS_RTOL * np.abs(ol)), (loss, ol)
    assert_close(gx, ogx, GRAD_RTOL, GRAD_ATOL, "normalized grad_x")
    assert_close(gy, ogy, GRAD_RTOL, GRAD_ATOL, "normalized grad_y")


def test_normalized_of_equal_inputs_is_zero():
    x, _ = synth.iid_normal_pair(2, 50, 50, 3, 97)
    loss, gx, gy = run_normalized(x, x.copy(), 1.0, 1, [1.0, 1.0])
    s = np.abs(oracle.batch(x, x, 1.0)[0])
    assert np.all(np.abs(loss) <= 1e-4 * np.maximum(1.0, s)), loss
    gscale = np.abs(oracle.batch(x, x, 1.0, grad_loss=np.ones(2))[1]).max()
    assert np.abs(gx).max() <= 1e-3 * gscale and np.abs(gy).max() <= 1e-3 * gscale


def run_normalized_unequal(x, y, gamma, mode, gl):
    L = _lib()
    xt, yt = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    B, N, D = x.shape
    M = y.shape[1]
    ws = L.workspace(L.OP_NORMALIZED_UNEQUAL, B, N, M, D, mode)
    loss = torch.empty(B, device="cuda")
    g = torch.tensor(np.asarray(gl, np.float32), device="cuda")
    gx, gy = torch.empty_like(xt), torch.empty_like(yt)
    L.sdtw_normalized_unequal(xt, yt, gamma, mode, loss, g, gx, gy, ws)
    assert L.sdtw_last_device_status(ws) == 0
    return loss.cpu().numpy().astype(np.float64), gx.cpu().numpy(), gy.cpu().numpy()


@pytest.mark.parametrize("mname,mode", MODES + [("unfused+extended", 2), ("fused+extended", 3)])
@pytest.mark.parametrize("N,M,D", [(100, 37, 8), (33, 130, 3), (1, 9, 2)])
def test_unequal_normalized_matches_oracle(mname, mode, N, M, D):
    x, y = synth.iid_normal_pair(3, N, M, D, 98, repeat=N * 1000 + M)
    gl = np.array(WEIGHTS_O1 if mode & 2 else mean_weights(3))
    loss, gx, gy = run_normalized_unequal(x, y, 0.8, mode, gl)
    ol, ogx, ogy = oracle.normalized_unequal(x, y, 0.8, grad_loss=gl)
    sxx = oracle.batch(x, x, 0.8)[0]
    syy = oracle.batch(y, y, 0.8)[0]
    atol = 1e-4 * np.maximum(1.0, np.maximum(np.abs(sxx), np.abs(syy)))
    assert np.all(np.abs(loss - ol) <= atol + LOSS_RTOL * np.abs(ol)), (loss, ol)
    assert_close(gx, ogx, GRAD_RTOL, GRAD_ATOL, f"unequal normalized {mname} grad_x")
    assert_close(gy, ogy, GRAD_RTOL, GRAD_ATOL, f"unequal normalized {mname} grad_y")


@pytest.mark.parametrize("mname,mode", MODES)
def test_unequal_normalized_at_equal_lengths_agrees_with_the_batched_entry(mname, mode):
    x, y = synth.iid_normal_pair(4, 64, 64, 5, 99)
    gl = [0.25, -0.5, 1.0, 0.125]
    a = run_normalized(x, y, 0.9, mode, gl)
    b = run_normalized_unequal(x, y, 0.9, mode, gl)
    scale = np.abs(oracle.batch(x, x, 0.9)[0]).max()
    assert np.abs(a[0] - b[0]).max() <= 1e-5 * max(1.0, scale)
    for u, v in zip(a[1:], b[1:]):
        assert np.abs(u - v).max() <= 1e-5 * max(1e-3, np.abs(u).max())


def test_unequal_normalized_through_autograd():
    from differentiable_series_alignment_gb300 import SoftDTW
    x, y = synth.iid_normal_pair(2, 40, 70, 4, 100)
    xt = torch.from_numpy(x).cuda().requires_grad_(True)
    yt = torch.from_numpy(y).cuda().requires_grad_(True)
    loss = SoftDTW(gamma=1.0, normalize=True, fused=True)(xt, yt)
    (loss * torch.tensor([0.5, -1.0], device="cuda")).sum().backward()
    ol, ogx, ogy = oracle.normalized_unequal(x, y, 1.0, grad_loss=[0.5, -1.0])
    s = np.maximum(np.abs(oracle.batch(x, x, 1.0)[0]), np.abs(oracle.batch(y, y, 1.0)[0]))
    assert np.all(np.abs(loss.detach().cpu().numpy() - ol) <= 1e-4 * np.maximum(1.0, s) + LOSS_RTOL * np.abs(ol))
    assert_close(xt.grad.cpu().numpy(), ogx, GRAD_RTOL, GRAD_ATOL, "autograd unequal normalized grad_x")
    assert_close(yt.grad.cpu().numpy(), ogy, GRAD_RTOL, GRAD_ATOL, "autograd unequal normalized grad_y")


CKPT = 1 | 4   # SDTW_FUSED | SDTW_CHECKPOINT


@pytest.mark.parametrize("N,M,D", [(64, 70, 8), (128, 33, 16), (129, 100, 5), (300, 77, 64)])
def test_checkpointed_fused_matches_oracle(N, M, D):
    # the checkpointed mode is fp32 only: batches of 32 at their own mean (D > 4)
    x, y = synth.iid_normal_pair(32, N, M, D, 101, repeat=N * 1000 + M)
    check_against_oracle(x, y, 0.9, CKPT, grad_loss=mean_weights(32), what=f"checkpoint {N}x{M}x{D}")


@pytest.mark.parametrize("mname,mode", [("fused+checkpoint", 5)])
def test_checkpointed_headline_config(mname, mode):
    # the headline workload's own inputs in the checkpointed mode (its results equal
    # the stored-state fused mode's bit for bit, see below)
    c = synth.WORKLOADS["headline"]
    x, y = synth.iid_normal_pair(c["B"], c["N"], c["M"], c["D"], c["seed"])
    check_against_oracle(x, y, 1.0, mode, what=f"headline {mname}")


@pytest.mark.parametrize("N,M", [(300, 77), (257, 130)])
def test_checkpointed_fused_agrees_with_stored_state(N, M):
    """The recomputed bands repeat the forward's arithmetic exactly, so losses and
    grad_x equal those of the stored-state fused mode bit for bit; grad_y sums the
    bands' terms in another order."""
    x, y = synth.iid_normal_pair(4, N, M, 12, 102, repeat=N)
    w = [0.03, -0.02, 0.05, 0.01]
    a = run_cuda(x, y, 1.1, 1, grad_loss=w)
    b = run_cuda(x, y, 1.1, CKPT, grad_loss=w)
    assert np.array_equal(a["loss"], b["loss"])
    assert np.array_equal(a["gx"], b["gx"])
    assert_close(b["gy"], a["gy"], 1e-5, 1e-8, "checkpoint grad_y vs stored state")


def test_checkpointed_padded_batch_and_autograd():
    from differentiable_series_alignment_gb300 import SoftDTW
    L = _lib()
    B, N, M, D, gamma = 3, 200, 150, 6, 0.8
    lx, ly = [200, 131, 7], [150, 90, 150]
    x, y = synth.iid_normal_pair(B, N, M, D, 103)
    for b in range(B):
        x[b, lx[b]:] = 0.0
        y[b, ly[b]:] = 0.0
    xt = torch.from_numpy(x).cuda().requires_grad_(True)
    yt = torch.from_numpy(y).cuda().requires_grad_(True)
    lxt = torch.tensor(lx, dtype=torch.int32, device="cuda")
    lyt = torch.tensor(ly, dtype=torch.int32, device="cuda")
    loss = SoftDTW(gamma=gamma, fused=True, checkpoint=True)(xt, yt, lxt, lyt)
    W = mean_weights(B)
    w = torch.tensor(W, device="cuda")
    (loss * w).sum().backward()
    loss = loss.detach().cpu().numpy()
    gx, gy = xt.grad.cpu().numpy(), yt.grad.cpu().numpy()
    for b in range(B):
        o = oracle.single(x[b, :lx[b]], y[b, :ly[b]], gamma, g=W[b])
        assert_close(loss[b:b + 1], [o["loss"]], LOSS_RTOL, 1e-6, f"checkpoint padded pair {b} loss")
        assert_close(gx[b, :lx[b]], o["gx"], GRAD_RTOL, GRAD_ATOL, f"checkpoint padded pair {b} grad_x")
        assert_close(gy[b, :ly[b]], o["gy"], GRAD_RTOL, GRAD_ATOL, f"checkpoint padded pair {b} grad_y")
        assert not np.any(gx[b, lx[b]:]) and not np.any(gy[b, ly[b]:])


# --------------------------------------------------------------------------- barycenter

@pytest.mark.parametrize("mname,mode", MODES)
def test_barycenter_steps_match_oracle(mname, mode):
    L = _lib()
    X = synth.block_waves(8, 96, 3, 4)
    z0 = X.astype(np.float64).mean(axis=0).astype(np.float32)
    Xt = torch.from_numpy(X).cuda()
    z = torch.from_numpy(z0.copy()).cuda()
    m = torch.zeros_like(z)
    v = torch.zeros_like(z)
    ws = L.workspace(L.OP_BARYCENTER, 8, 96, 96, 3, mode)
    lo = torch.empty(1, device="cuda")
    zo, mo, vo = z0.astype(np.float64), np.zeros_like(z0, np.float64), np.zeros_like(z0, np.float64)
    for t in (1, 2, 3):
        # oracle step from the CUDA path's current state, so the comparison is per step
        zc, mc, vc = z.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
        zo, mo, vo, lref, _ = oracle.barycenter_step(zc, mc, vc, t, X, 1.0, lr=0.1)
        L.sdtw_barycenter_step(z, m, v, t, Xt, 1.0, 0.1, 0.9, 0.999, 1e-8, mode, lo, ws)
        assert L.sdtw_last_device_status(ws) == 0
        assert_close(lo.cpu().numpy(), [lref], LOSS_RTOL, 0.0, f"step {t} loss")
        assert_close(m.cpu().numpy(), mo, GRAD_RTOL, GRAD_ATOL, f"step {t} first moment")
        # z moves by ~lr per coordinate; compare the update itself
        assert_close(z.cpu().numpy() - zc, zo - zc, 2e-3, 1e-6, f"step {t} update")


# --------------------------------------------------------------------------- padded batches

@pytest.mark.parametrize("mname,mode,weights", [("unfused", 0, mean_weights(4)),
                                                ("fused", 1, mean_weights(4)),
                                                ("unfused+extended", 2, WEIGHTS_O1 + [0.25]),
                                                ("fused+extended", 3, WEIGHTS_O1 + [0.25])])
def test_padded_batch_matches_oracle(mname, mode, weights):
    L = _lib()
    B, N, M, D, gamma = 4, 100, 90, 6, 0.9
    lx, ly = [100, 37, 1, 64], [90, 90, 5, 33]
    x, y = synth.iid_normal_pair(B, N, M, D, 99)
    for b in range(B):               # zero padding beyond each pair's lengths
        x[b, lx[b]:] = 0.0
        y[b, ly[b]:] = 0.0
    xt, yt = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    lxt = torch.tensor(lx, dtype=torch.int32, device="cuda")
    lyt = torch.tensor(ly, dtype=torch.int32, device="cuda")
    ws = L.workspace(L.OP_FWD_BWD, B, N, M, D, mode)
    loss = torch.empty(B, device="cuda")
    gx, gy = torch.empty_like(xt), torch.empty_like(yt)
    g = torch.tensor(weights, dtype=torch.float32, device="cuda")
    L.sdtw_forward_varlen(xt, yt, lxt, lyt, gamma, mode, loss, ws)
    L.sdtw_backward_varlen(xt, yt, lxt, lyt, gamma, mode, g, gx, gy, ws)
    assert L.sdtw_last_device_status(ws) == 0
    loss, gx, gy = loss.cpu().numpy(), gx.cpu().numpy(), gy.cpu().numpy()
    for b in range(B):
        o = oracle.single(x[b, :lx[b]], y[b, :ly[b]], gamma, g=weights[b])
        assert_close(loss[b:b + 1], [o["loss"]], LOSS_RTOL, 1e-6, f"padded {mname} pair {b} loss")
        assert_close(gx[b, :lx[b]], o["gx"], GRAD_RTOL, GRAD_ATOL, f"padded {mname} pair {b} grad_x")
        assert_close(gy[b, :ly[b]], o["gy"], GRAD_RTOL, GRAD_ATOL, f"padded {mname} pair {b} grad_y")
        assert not np.any(gx[b, lx[b]:]) and not np.any(gy[b, ly[b]:])   # padding gets zero gradient


def test_padded_batch_autograd_and_full_lengths():
    from differentiable_series_alignment_gb300 import SoftDTW
    x, y = synth.iid_normal_pair(3, 50, 41, 4, 100)
    xt = torch.from_numpy(x).cuda().requires_grad_(True)
    yt = torch.from_numpy(y).cuda()
    full = SoftDTW(gamma=1.0)(xt, yt)
    lens = SoftDTW(gamma=1.0)(xt, yt, torch.tensor([50, 50, 50]), torch.tensor([41, 41, 41]))
    assert_close(lens.detach().cpu().numpy(), full.detach().cpu().numpy(), 1e-6, 0.0, "full lengths")
    lens.sum().backward()
    assert torch.isfinite(xt.grad).all()


# --------------------------------------------------------------------------- caller-supplied costs

def _cost_batch(kind, B, N, M, seed):
    g = np.random.default_rng(seed)
    if kind == "l1":      # |x - y| summed over 3 features: a non-Euclidean, non-negative cost
        x = g.standard_normal((B, N, 3))
        y = g.standard_normal((B, M, 3))
        return np.abs(x[:, :, None, :] - y[:, None, :, :]).sum(-1).astype(np.float32)
    return (2.0 * g.standard_normal((B, N, M))).astype(np.float32)   # signed costs


@pytest.mark.parametrize("mname,mode,weights", [("fp32", 0, mean_weights(3)), ("extended", 2, WEIGHTS_O1)])
@pytest.mark.parametrize("kind", ["l1", "signed"])
@pytest.mark.parametrize("N,M", [(1, 1), (1, 9), (7, 1), (33, 31), (100, 37), (129, 130)])
def test_given_cost_matches_oracle(mname, mode, weights, kind, N, M):
    L = _lib()
    B, gamma = 3, 0.8
    C = _cost_batch(kind, B, N, M, N * 1000 + M)
    Ct = torch.from_numpy(C).cuda()
    ws = L.workspace(L.OP_COST, B, N, M, 1, mode)
    loss = torch.empty(B, device="cuda")
    gC = torch.empty_like(Ct)
    g = torch.tensor(weights, dtype=torch.float32, device="cuda")
    L.sdtw_forward_cost(Ct, gamma, mode, loss, ws)
    L.sdtw_backward_cost(Ct, gamma, mode, g, gC, ws)
    assert L.sdtw_last_device_status(ws) == 0
    ol, ogC = [], []
    for b in range(B):
        R = oracle.forward_from_cost(C[b], gamma)
        ol.append(R[N, M])
        ogC.append(weights[b] * oracle.backward_from_cost(C[b], R, gamma))
    assert_close(loss.cpu().numpy(), np.array(ol), LOSS_RTOL, 1e-6, f"cost {kind} {N}x{M} {mname} loss")
    assert_close(gC.cpu().numpy(), np.stack(ogC), GRAD_RTOL, GRAD_ATOL, f"cost {kind} {N}x{M} {mname} grad_C")


def test_given_squared_euclidean_cost_reproduces_softdtw():
    # the cost path fed the squared Euclidean cost equals the x/y path, values and
    # (through the chain rule dC/dx) gradients, via the autograd wrappers
    from differentiable_series_alignment_gb300 import SoftDTW, soft_dtw_cost
    x, y = synth.iid_normal_pair(4, 70, 61, 5, 97)
    xt = torch.from_numpy(x).cuda().requires_grad_(True)
    yt = torch.from_numpy(y).cuda().requires_grad_(True)
    a = SoftDTW(gamma=0.9)(xt, yt)
    a.mean().backward()
    gxa = xt.grad.detach().clone()
    xt.grad = None
    C = ((xt[:, :, None, :] - yt[:, None, :, :]) ** 2).sum(-1)   # test-side cost, plain torch
    b = soft_dtw_cost(C, gamma=0.9)
    b.mean().backward()
    assert_close(b.detach().cpu().numpy(), a.detach().cpu().numpy(), LOSS_RTOL, 0.0, "cost vs x/y loss")
    assert_close(xt.grad.cpu().numpy(), gxa.cpu().numpy(), GRAD_RTOL, GRAD_ATOL, "cost vs x/y grad_x")


@pytest.mark.parametrize("mname,mode", MODES)
def test_clipped_barycenter_steps_match_oracle(mname, mode):
    # a bound well below ||g|| so the clipping acts on every step
    L = _lib()
    X = synth.block_waves(8, 96, 3, 5)
    z0 = X.astype(np.float64).mean(axis=0).astype(np.float32)
    Xt = torch.from_numpy(X).cuda()
    z = torch.from_numpy(z0.copy()).cuda()
    m, v = torch.zeros_like(z), torch.zeros_like(z)
    ws = L.workspace(L.OP_BARYCENTER, 8, 96, 96, 3, mode)
    lo = torch.empty(1, device="cuda")
    _, _, _, _, g0 = oracle.barycenter_step(z0, np.zeros_like(z0), np.zeros_like(z0), 1, X, 1.0)
    clip = 0.3 * float(np.linalg.norm(g0))
    for t in (1, 2, 3):
        zc, mc, vc = z.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
        zo, mo, vo, lref, _ = oracle.barycenter_step(zc, mc, vc, t, X, 1.0, lr=0.1, max_grad_norm=clip)
        L.sdtw_barycenter_step_clipped(z, m, v, t, Xt, 1.0, 0.1, 0.9, 0.999, 1e-8, clip, mode, lo, ws)
        assert L.sdtw_last_device_status(ws) == 0
        assert_close(lo.cpu().numpy(), [lref], LOSS_RTOL, 0.0, f"clipped step {t} loss")
        assert_close(m.cpu().numpy(), mo, GRAD_RTOL, GRAD_ATOL, f"clipped step {t} first moment")
        assert_close(v.cpu().numpy(), vo, 2e-3, 1e-9, f"clipped step {t} second moment")
        assert_close(z.cpu().numpy() - zc, zo - zc, 2e-3, 1e-6, f"clipped step {t} update")


def test_barycenter_driver_schedule_clipping_and_early_stopping():
    from differentiable_series_alignment_gb300 import softdtw_barycenter
    X = torch.from_numpy(synth.block_waves(16, 128, 2, 6)).cuda()
    z, lo = softdtw_barycenter(X, gamma=1.0, max_iter=400, lr=0.1, lr_schedule="cosine", lr_min=0.001,
                               max_grad_norm=1.0, early_stopping=True, tol=1e-3, patience=20, check_every=10,
                               return_losses=True)
    lo = lo.cpu().numpy()
    assert np.all(np.isfinite(lo)) and torch.isfinite(z).all()
    assert len(lo) < 400            # converged and stopped early
    assert lo[-1] < lo[0]
    z2, lo2 = softdtw_barycenter(X, gamma=1.0, max_iter=30, lr=0.1, return_losses=True)
    assert len(lo2) == 30


# --------------------------------------------------------------------------- device status

@pytest.mark.parametrize("mname,mode", MODES + [("unfused+extended", 2), ("fused+extended", 3)])
@pytest.mark.parametrize("B,chunks", [(5, 3), (1, 4), (7, 8), (32, 3)])
def test_host_batch_matches_oracle_and_device_path(mname, mode, B, chunks):
    """Host buffers in, host buffers out, the batch cut into uneven chunks on side
    streams: the same losses and gradients as the oracle and the device-buffer path.
    Weights: the batch's own mean (fp32 takes the batch of 32 only, D = 8 > 4),
    O(1) in the double-float mode."""
    L = _lib()
    if not (mode & 2) and B < 32:
        pytest.skip("fp32 state: batch-mean weights of a batch below 32 pairs at D > 4 need the double-float mode")
    N, M, D, gamma = 100, 77, 8, 0.8
    x, y = synth.iid_normal_pair(B, N, M, D, 77, repeat=B * 10 + chunks)
    w = np.array(mean_weights(B)) if not (mode & 2) else np.array([WEIGHTS_O1[b % 3] for b in range(B)])
    xh, yh = torch.from_numpy(x).pin_memory(), torch.from_numpy(y).pin_memory()
    gl = torch.from_numpy(w.astype(np.float32)).pin_memory()
    loss = torch.full((B,), float("nan")).pin_memory()
    gx, gy = torch.full_like(xh, float("nan")).pin_memory(), torch.full_like(yh, float("nan")).pin_memory()
    ws = L.host_workspace(B, N, M, D, mode, chunks)
    L.sdtw_value_and_grad_host(xh, yh, gl, gamma, mode, loss, gx, gy, chunks, ws)
    assert L.sdtw_last_device_status(ws) == 0
    ol, ogx, ogy = oracle.batch(x, y, gamma, grad_loss=w)
    assert_close(loss.numpy(), ol, LOSS_RTOL, 0.0, f"host batch {mname} loss")
    assert_close(gx.numpy(), ogx, GRAD_RTOL, GRAD_ATOL, f"host batch {mname} grad_x")
    assert_close(gy.numpy(), ogy, GRAD_RTOL, GRAD_ATOL, f"host batch {mname} grad_y")
    dev = run_cuda(x, y, gamma, mode, grad_loss=w)
    assert_close(loss.numpy(), dev["loss"], 1e-6, 0.0, f"host batch {mname} loss vs device path")
    assert np.array_equal(gx.numpy(), dev["gx"].astype(np.float32))
    assert np.array_equal(gy.numpy(), dev["gy"].astype(np.float32))


def test_host_batch_high_level_function_and_loss_only():
    from differentiable_series_alignment_gb300 import value_and_grad_host
    L = _lib()
    B, N, M, D = 6, 64, 48, 5
    x, y = synth.iid_normal_pair(B, N, M, D, 78)
    loss, gx, gy = value_and_grad_host(torch.from_numpy(x), torch.from_numpy(y), gamma=1.0, fused=True,
                                       grad_loss=torch.full((B,), 1.0 / B), chunks=4)
    ol, ogx, ogy = oracle.batch(x, y, 1.0, grad_loss=np.full(B, 1.0 / B))
    assert_close(loss.numpy(), ol, LOSS_RTOL, 0.0, "value_and_grad_host loss")
    assert_close(gx.numpy(), ogx, GRAD_RTOL, GRAD_ATOL, "value_and_grad_host grad_x")
    assert_close(gy.numpy(), ogy, GRAD_RTOL, GRAD_ATOL, "value_and_grad_host grad_y")
    # loss only: no gradients asked for, grad_loss may be absent
    ws = L.host_workspace(B, N, M, D, L.UNFUSED, 2)
    lo = torch.empty(B).pin_memory()
    L.sdtw_value_and_grad_host(torch.from_numpy(x), torch.from_numpy(y), None, 1.0, L.UNFUSED, lo, None, None, 2, ws)
    assert L.sdtw_last_device_status(ws) == 0
    assert_close(lo.numpy(), ol, LOSS_RTOL, 0.0, "host batch loss only")


def test_high_level_api_picks_the_precision_the_weights_need():
    """Through the public API the precision follows the upstream weights: at the
    shape where the fp32 state misses abs 1e-5 for a batch of 3 (70 x 91, D = 20,
    gamma = 0.8), SoftDTW(...).mean() over B = 3 and value_and_grad_host with O(1)
    weights both select the double-float state and hold the tolerance."""
    from differentiable_series_alignment_gb300 import SoftDTW, value_and_grad_host
    L = _lib()
    B, gamma = 3, 0.8
    x, y = synth.iid_normal_pair(B, 70, 91, 20, 96)
    assert L.auto_precision(gamma, 70, 91, 20, B) == L.EXTENDED
    ol, ogx, ogy = oracle.batch(x, y, gamma, grad_loss=np.full(B, 1.0 / B))
    for fused in (False, True):
        xt = torch.from_numpy(x).cuda().requires_grad_(True)
        yt = torch.from_numpy(y).cuda().requires_grad_(True)
        loss = SoftDTW(gamma=gamma, fused=fused)(xt, yt)
        loss.mean().backward()
        assert_close(loss.detach().cpu().numpy(), ol, LOSS_RTOL, 0.0, f"api mean loss fused={fused}")
        assert_close(xt.grad.cpu().numpy(), ogx, GRAD_RTOL, GRAD_ATOL, f"api mean grad_x fused={fused}")
        assert_close(yt.grad.cpu().numpy(), ogy, GRAD_RTOL, GRAD_ATOL, f"api mean grad_y fused={fused}")
    w = np.array(WEIGHTS_O1)
    loss, gx, gy = value_and_grad_host(torch.from_numpy(x), torch.from_numpy(y), gamma=gamma,
                                       grad_loss=torch.from_numpy(w.astype(np.float32)))
    ol, ogx, ogy = oracle.batch(x, y, gamma, grad_loss=w)
    assert_close(loss.numpy(), ol, LOSS_RTOL, 0.0, "api O(1) weights loss")
    assert_close(gx.numpy(), ogx, GRAD_RTOL, GRAD_ATOL, "api O(1) weights grad_x")
    assert_close(gy.numpy(), ogy, GRAD_RTOL, GRAD_ATOL, "api O(1) weights grad_y")


def test_withheld_ready_flag_times_out_and_recovers():
    L = _lib()
    x, y = synth.iid_normal_pair(2, 160, 40, 3, 98)
    xt, yt = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    ws = L.workspace(L.OP_FWD_BWD, 2, 160, 40, 3, 1)
    loss = torch.empty(2, device="cuda")
    try:
        with warps(1):
            L.sdtw_debug_set_wait(0.05, skip_publish=True)
            L.sdtw_forward(xt, yt, 1.0, 1, loss, ws)
            assert L.sdtw_last_device_status(ws) == 7   # SDTW_ERR_TIMEOUT
    finally:
        L.sdtw_debug_set_wait(0.0, skip_publish=False)
    # the context is still usable and the next call is correct
    got = run_cuda(x, y, 1.0, 1)
    ol, _, _ = oracle.batch(x, y, 1.0)
    assert_close(got["loss"], ol, LOSS_RTOL, 0.0, "after timeout")


def test_validation_errors_raise():
    L = _lib()
    x = torch.zeros((2, 5, 3), device="cuda")
    ws = L.workspace(L.OP_FWD_BWD, 2, 5, 5, 3, 0)
    loss = torch.empty(2, device="cuda")
    with pytest.raises(L.SdtwError) as e:
        L.sdtw_forward(x, x, 0.0, 0, loss, ws)
    assert e.value.code == 2
    with pytest.raises(L.SdtwError) as e:
        L.sdtw_forward(x, x, 1.0, 0, loss, ws[:100])
    assert e.value.code == 5


# The library's calls can be captured into a CUDA graph (the timed step of the
# benchmark replays one): launches, memsets and the side-stream forks and joins of a
# forward + backward, replayed, give the eager results bit for bit.
@pytest.mark.parametrize("mode", [0, 1, 2, 3, 5])
def test_graph_capture_replays_the_eager_results(mode):
    L = _lib()
    x, y = synth.iid_normal_pair(4, 150, 130, 16, 107)
    xt, yt = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    ws = L.workspace(L.OP_FWD_BWD, 4, 150, 130, 16, mode)
    g = torch.tensor(mean_weights(4), dtype=torch.float32, device="cuda")
    loss, gx, gy = torch.empty(4, device="cuda"), torch.empty_like(xt), torch.empty_like(yt)

    def fwd_bwd():
        L.sdtw_forward(xt, yt, 0.8, mode, loss, ws)
        L.sdtw_backward(xt, yt, 0.8, mode, g, gx, gy, ws)

    fwd_bwd()
    assert L.sdtw_last_device_status(ws) == 0
    ref = [t.clone() for t in (loss, gx, gy)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd_bwd()
    for t in (loss, gx, gy):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert L.sdtw_last_device_status(ws) == 0
    for a, b in zip((loss, gx, gy), ref):
        assert torch.equal(a, b)
