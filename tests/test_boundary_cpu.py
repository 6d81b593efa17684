"""The C ABI without a GPU: the library loads, exports every declared symbol,
sizes workspaces, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from helpers import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "sdtw.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sdtw_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from differentiable_series_alignment_gb300 import _lib
    return _lib.load()


def test_header_declares_the_documented_entry_points():
    names = _declared_functions()
    for n in ("sdtw_workspace_bytes", "sdtw_forward", "sdtw_backward", "sdtw_normalized",
              "sdtw_barycenter_step", "sdtw_last_device_status", "sdtw_status_string", "sdtw_distance"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from differentiable_series_alignment_gb300 import _lib
    for n in _declared_functions():
        assert hasattr(lib, n), f"libsdtw.so does not export {n}"
    assert set(_declared_functions()) == set(_lib.EXPORTS)


def test_workspace_sizes(lib):
    from differentiable_series_alignment_gb300 import _lib as L
    u = L.sdtw_workspace_bytes(L.OP_FWD_BWD, 32, 512, 512, 64, L.UNFUSED)
    f = L.sdtw_workspace_bytes(L.OP_FWD_BWD, 32, 512, 512, 64, L.FUSED)
    # skewed slots: 16 blocks x (512+31 rounded up to a multiple of 16) x 32 per problem
    slots = 32 * 16 * 544 * 32
    # tensor-core cost operands in both modes: x and y images (three bf16 parts, one
    # K-block of 64 features, rows padded to 128) and row norms (hi, lo)
    simg = 2 * (32 * 1 * 3 * 512 * 128) + 2 * (32 * 512 * 4)
    assert f >= slots * (8 + 4) + simg   # (vl,hu) pairs + alignment matrix
    assert u >= f + slots * 4            # + the stored cost tensor
    assert u - f < slots * 4 + 4096
    # pre-split [Y|1] and [X|1] operand images of the gradient contraction: per
    # problem and K-tile of 32, hi + lo tiles of roundup(D+1, 16) rows x 128 bytes
    bimg = 2 * 32 * (512 // 32) * 2 * 80 * 128
    assert f >= slots * (8 + 4) + bimg
    n = L.sdtw_workspace_bytes(L.OP_NORMALIZED, 32, 512, 999, 64, L.FUSED)   # M ignored
    assert n >= 3 * (f - bimg) + bimg - 3 * 4096   # three batches of state, one set of images
    assert L.sdtw_workspace_bytes(L.OP_BARYCENTER, 64, 1024, 1024, 8, L.FUSED) > 0
    for bad in [(0, 4, 4, 4), (4, 0, 4, 4), (4, 4, 0, 4), (4, 4, 4, 0)]:
        assert L.sdtw_workspace_bytes(L.OP_FWD_BWD, *bad, L.UNFUSED) == 0
    assert L.sdtw_workspace_bytes(7, 4, 4, 4, 4, L.UNFUSED) == 0
    assert L.sdtw_workspace_bytes(L.OP_FWD_BWD, 4, 4, 4, 4, 4) == 0
    # extended precision: 16-byte log-probabilities instead of 8-byte pairs; unfused
    # also stores the double-float cost (8 bytes). Both modes carry the exact
    # tensor-core costs' digit images (five bf16 slices per K-block of 64 up to
    # D = 128, six above, up to D = 400) and row info
    fx = L.sdtw_workspace_bytes(L.OP_FWD_BWD, 32, 512, 512, 64, L.FUSED | L.EXTENDED)
    ux = L.sdtw_workspace_bytes(L.OP_FWD_BWD, 32, 512, 512, 64, L.UNFUSED | L.EXTENDED)
    oimg = 2 * (32 * 1 * 5 * 512 * 128) + 2 * (32 * 512 * 16)
    assert fx - (f - bimg - simg) >= slots * 8 + oimg and ux - fx >= slots * 8
    fx256 = L.sdtw_workspace_bytes(L.OP_FWD_BWD, 32, 512, 512, 256, L.FUSED | L.EXTENDED)
    ux256 = L.sdtw_workspace_bytes(L.OP_FWD_BWD, 32, 512, 512, 256, L.UNFUSED | L.EXTENDED)
    oimg256 = 2 * (32 * 4 * 6 * 512 * 128) + 2 * (32 * 512 * 16)
    assert ux256 - fx256 >= slots * 8 and fx256 >= slots * (16 + 4) + oimg256


def _fwd(lib, x=0x1000, y=0x2000, B=2, N=3, M=4, D=2, gamma=1.0, mode=0, loss=0x3000, ws=0x100000,
         ws_bytes=1 << 40):
    vp = ctypes.c_void_p
    return lib.sdtw_forward(vp(x) if x else None, vp(y) if y else None, B, N, M, D, gamma, mode,
                            vp(loss) if loss else None, vp(ws) if ws else None, ws_bytes, None)


def test_validation_codes_need_no_device(lib):
    # Every case below must fail in host-side validation, before any CUDA call.
    assert _fwd(lib, B=0) == 3            # SDTW_ERR_EMPTY
    assert _fwd(lib, N=0) == 3
    assert _fwd(lib, M=0) == 3
    assert _fwd(lib, D=0) == 3
    assert _fwd(lib, gamma=0.0) == 2      # SDTW_ERR_GAMMA
    assert _fwd(lib, gamma=-1.0) == 2
    assert _fwd(lib, gamma=float("inf")) == 2
    assert _fwd(lib, gamma=float("nan")) == 2
    assert _fwd(lib, mode=4) == 1         # SDTW_ERR_ARG
    assert _fwd(lib, x=0) == 1
    assert _fwd(lib, loss=0) == 1
    assert _fwd(lib, ws=0) == 5           # SDTW_ERR_WORKSPACE
    assert _fwd(lib, ws=0x100010) == 5    # misaligned
    assert _fwd(lib, ws_bytes=16) == 5    # too small
    assert _fwd(lib, D=100000) == 8       # SDTW_ERR_TOO_LARGE


def test_status_strings(lib):
    for code in range(9):
        assert lib.sdtw_status_string(code)
    assert b"gamma" in lib.sdtw_status_string(2)


def test_normalized_and_barycenter_validation(lib):
    vp = ctypes.c_void_p
    # gamma invalid
    assert lib.sdtw_normalized(vp(0x1000), vp(0x2000), 2, 3, 2, 0.0, 0, vp(0x3000), None, None, None,
                               vp(0x100000), 1 << 40, None) == 2
    # t = 0 is not a valid Adam step
    assert lib.sdtw_barycenter_step(vp(0x1000), vp(0x2000), vp(0x3000), 0, vp(0x4000), 4, 8, 8, 2, 1.0, 0.1,
                                    0.9, 0.999, 1e-8, 1, None, vp(0x100000), 1 << 40, None) == 1
    # empty sequences
    assert lib.sdtw_barycenter_step(vp(0x1000), vp(0x2000), vp(0x3000), 1, vp(0x4000), 0, 8, 8, 2, 1.0, 0.1,
                                    0.9, 0.999, 1e-8, 1, None, vp(0x100000), 1 << 40, None) == 3


def test_auto_precision_rule():
    from differentiable_series_alignment_gb300 import _lib as L
    assert L.auto_precision(1.0, 512, 512, 64) == 0            # the headline shape stays fp32
    assert L.auto_precision(1.0, 512, 512) == 0
    assert L.auto_precision(1.0, 512, 512, 65) == L.EXTENDED     # wide features
    assert L.auto_precision(0.01, 64, 64, 4) == L.EXTENDED      # small gamma
    assert L.auto_precision(1.0, 4096, 8, 4) == L.EXTENDED      # long sequences
    assert L.auto_precision(1.0, 8, 4095, 4) == 0
    # batch rule: fp32 for batch-mean losses over B >= 32 pairs, or D <= 4
    assert L.auto_precision(1.0, 512, 512, 64, 32) == 0          # the headline batch
    assert L.auto_precision(1.0, 512, 512, 64, 31) == L.EXTENDED
    assert L.auto_precision(1.0, 64, 64, 4, 4) == 0              # the small workload
    assert L.auto_precision(1.0, 64, 64, 5, 4) == L.EXTENDED
    assert L.auto_precision(1.0, 1024, 1024, 8, 64) == 0         # the barycenter workload (mean over K=64)
    assert L.auto_precision(1.0, 128, 128, 20, None) == 0        # no batch rule without B
    assert L.auto_precision(1.0, 256, 256, 128, 32) == L.EXTENDED  # wide features: double-float state
    assert L.auto_precision(1.0, 8192, 8192, 128, 8) == L.EXTENDED  # the long workload


def test_given_cost_entry_points_validate_on_the_host(lib):
    from differentiable_series_alignment_gb300 import _lib as L
    # workspace: the DP state of an unfused problem without x/y operand images
    w = L.sdtw_workspace_bytes(L.OP_COST, 4, 100, 37, 0, L.UNFUSED)
    slots = 4 * 4 * 80 * 32    # 4 problems x 4 row blocks x T = 37 + 31 rounded up to 16 x 32 lanes
    assert w >= slots * (8 + 4 + 4)   # (v_left, h_up) pairs, alignment matrix, cost
    assert L.sdtw_workspace_bytes(L.OP_COST, 4, 100, 37, 7, L.UNFUSED) == w      # D is ignored
    assert L.sdtw_workspace_bytes(L.OP_COST, 4, 100, 37, 1, L.FUSED) == 0        # nothing to fuse
    assert L.sdtw_workspace_bytes(L.OP_COST, 4, 100, 37, 1, L.EXTENDED) > w
    vp = ctypes.c_void_p
    f = lib.sdtw_forward_cost
    f.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, vp, vp,
                  ctypes.c_size_t, vp]
    f.restype = ctypes.c_int
    ok = dict(C=vp(0x1000), B=2, N=3, M=4, g=1.0, mode=0, loss=vp(0x2000), ws=vp(0x100000), n=1 << 40)
    call = lambda **kw: f(*[dict(ok, **kw)[k] for k in ("C", "B", "N", "M", "g", "mode", "loss", "ws", "n")], None)
    assert call(B=0) == 3 and call(M=0) == 3          # SDTW_ERR_EMPTY
    assert call(g=0.0) == 2 and call(g=float("nan")) == 2
    assert call(mode=L.FUSED) == 1 and call(mode=4) == 1
    assert call(C=None) == 1 and call(loss=None) == 1
    assert call(ws=None) == 5 and call(ws=vp(0x100001)) == 5 and call(n=16) == 5


def test_cosine_schedule_values():
    from differentiable_series_alignment_gb300 import cosine_lr
    assert cosine_lr(1, 100, 0.1) == 0.1                                      # starts at lr
    assert cosine_lr(51, 100, 0.1, 0.0) == pytest.approx(0.05)                # halfway: the mean
    assert cosine_lr(101, 100, 0.1, 0.01) == pytest.approx(0.01)              # ends at lr_min
    assert all(cosine_lr(t, 100, 0.1) >= cosine_lr(t + 1, 100, 0.1) for t in range(1, 100))


def test_host_batch_workspace_and_validation(lib):
    from differentiable_series_alignment_gb300 import _lib as L
    B, N, M, D = 32, 512, 512, 64
    io = 4 * (2 * B * N * D + 2 * B * M * D + 2 * B)      # x, y, grad_x, grad_y, grad_loss, loss
    for mode in (L.UNFUSED, L.FUSED):
        w4 = L.sdtw_host_workspace_bytes(B, N, M, D, mode, 4)
        per_chunk = L.sdtw_workspace_bytes(L.OP_FWD_BWD, B // 4, N, M, D, mode)
        assert w4 >= io + 4 * per_chunk
        assert w4 < io + 4 * per_chunk + 16 * 4096
        assert L.sdtw_host_workspace_bytes(B, N, M, D, mode, 0) == L.sdtw_host_workspace_bytes(B, N, M, D, mode, 2)
        assert L.sdtw_host_workspace_bytes(B, N, M, D, mode, 99) == L.sdtw_host_workspace_bytes(B, N, M, D, mode, 8)
        # chunks never exceed the batch; uneven chunks are sized for the largest
        assert L.sdtw_host_workspace_bytes(3, N, M, D, mode, 8) == L.sdtw_host_workspace_bytes(3, N, M, D, mode, 3)
        w5 = L.sdtw_host_workspace_bytes(5, N, M, D, mode, 2)
        assert w5 >= 2 * L.sdtw_workspace_bytes(L.OP_FWD_BWD, 3, N, M, D, mode)
    assert L.sdtw_host_workspace_bytes(0, N, M, D, L.UNFUSED, 4) == 0
    assert L.sdtw_host_workspace_bytes(B, N, M, 0, L.UNFUSED, 4) == 0
    vp = ctypes.c_void_p
    ok = dict(x=vp(0x1000), y=vp(0x2000), g=vp(0x3000), B=2, N=3, M=4, D=2, gamma=1.0, mode=0, loss=vp(0x4000),
              gx=vp(0x5000), gy=vp(0x6000), chunks=2, ws=vp(0x100000), n=1 << 40)
    keys = ("x", "y", "g", "B", "N", "M", "D", "gamma", "mode", "loss", "gx", "gy", "chunks", "ws", "n")
    call = lambda **kw: lib.sdtw_value_and_grad_host(*[dict(ok, **kw)[k] for k in keys], None)
    # every case fails in host-side validation, before any CUDA call
    assert call(B=0) == 3 and call(D=0) == 3             # SDTW_ERR_EMPTY
    assert call(gamma=0.0) == 2                          # SDTW_ERR_GAMMA
    assert call(x=None) == 1 and call(loss=None) == 1    # SDTW_ERR_ARG
    assert call(g=None) == 1                             # gradients asked for without grad_loss
    assert call(mode=4) == 1
    assert call(ws=None) == 5 and call(ws=vp(0x100008)) == 5 and call(n=64) == 5   # SDTW_ERR_WORKSPACE


def test_unequal_normalized_workspace_and_validation(lib):
    from differentiable_series_alignment_gb300 import _lib as L
    B, N, M, D = 4, 100, 37, 8
    for mode in (L.UNFUSED, L.FUSED, L.FUSED | L.EXTENDED):
        w = L.sdtw_workspace_bytes(L.OP_NORMALIZED_UNEQUAL, B, N, M, D, mode)
        parts = [L.sdtw_workspace_bytes(L.OP_FWD_BWD, B, n, m, D, mode) for n, m in ((N, M), (N, N), (M, M))]
        assert sum(parts) <= w <= sum(parts) + 3 * 256
    assert L.sdtw_workspace_bytes(L.OP_NORMALIZED_UNEQUAL, 0, N, M, D, L.UNFUSED) == 0
    assert L.sdtw_workspace_bytes(L.OP_NORMALIZED_UNEQUAL, B, N, 0, D, L.UNFUSED) == 0
    vp = ctypes.c_void_p
    ok = dict(x=vp(0x1000), y=vp(0x2000), B=2, N=5, M=3, D=2, g=1.0, mode=0, loss=vp(0x3000), gl=None, gx=None,
              gy=None, ws=vp(0x100000), n=1 << 40)
    keys = ("x", "y", "B", "N", "M", "D", "g", "mode", "loss", "gl", "gx", "gy", "ws", "n")
    call = lambda **kw: lib.sdtw_normalized_unequal(*[dict(ok, **kw)[k] for k in keys], None)
    # every case fails in host-side validation, before any CUDA call
    assert call(M=0) == 3 and call(B=0) == 3              # SDTW_ERR_EMPTY
    assert call(g=0.0) == 2                                # SDTW_ERR_GAMMA
    assert call(y=None) == 1 and call(loss=None) == 1 and call(mode=8) == 1
    assert call(ws=None) == 5 and call(ws=vp(0x100004)) == 5 and call(n=100) == 5


def test_checkpoint_workspace_and_validation(lib):
    from differentiable_series_alignment_gb300 import _lib as L
    B, N, M, D = 32, 512, 512, 64
    full = L.sdtw_workspace_bytes(L.OP_FWD_BWD, B, N, M, D, L.FUSED)
    ck = L.sdtw_workspace_bytes(L.OP_FWD_BWD, B, N, M, D, L.FUSED | L.CHECKPOINT)
    T = 544
    band = B * 4 * T * 32                       # cells of one 128-row band of every problem
    assert ck > 2 * band * 12                   # (v_left, h_up) pairs and E of two bands
    assert full - ck >= (B * 16 * T * 32 - 2 * band) * 12   # the other bands' state and E are gone
    assert ck < 0.6 * full
    # only the fp32 tensor-core fused path checkpoints
    assert L.sdtw_workspace_bytes(L.OP_FWD_BWD, B, N, M, D, L.UNFUSED | L.CHECKPOINT) == 0
    assert L.sdtw_workspace_bytes(L.OP_FWD_BWD, B, N, M, D, L.FUSED | L.EXTENDED | L.CHECKPOINT) == 0
    assert L.sdtw_workspace_bytes(L.OP_FWD_BWD, B, N, M, 65, L.FUSED | L.CHECKPOINT) == 0   # beyond the tensor-core width
    assert L.sdtw_workspace_bytes(L.OP_NORMALIZED, B, N, N, D, L.FUSED | L.CHECKPOINT) == 0
    assert L.sdtw_workspace_bytes(L.OP_FWD_BWD, 2, 3, 4, 2, 8) == 0
    # host-side validation, before any CUDA call
    assert _fwd(lib, mode=L.FUSED | L.CHECKPOINT, ws_bytes=16) == 5     # accepted flag, small workspace
    assert _fwd(lib, mode=L.UNFUSED | L.CHECKPOINT) == 1
    assert _fwd(lib, mode=L.FUSED | L.EXTENDED | L.CHECKPOINT) == 1
    assert _fwd(lib, mode=L.FUSED | L.CHECKPOINT, D=65) == 1
    vp = ctypes.c_void_p
    assert lib.sdtw_normalized(vp(0x1000), vp(0x2000), 2, 3, 2, 1.0, L.FUSED | L.CHECKPOINT, vp(0x3000), None,
                               None, None, vp(0x100000), 1 << 40, None) == 1
