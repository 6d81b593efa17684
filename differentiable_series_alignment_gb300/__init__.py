"""Batched Soft-DTW on GB300 (sm_103a): a C-ABI CUDA library and its binding.

Low level (same names as the C entry points, torch tensors for pointers):
    sdtw_workspace_bytes, sdtw_distance, sdtw_forward, sdtw_backward,
    sdtw_normalized, sdtw_barycenter_step, sdtw_last_device_status

High level, following the usage shown in the SoftDTW-CUDA (PyTorch + Numba)
README ("Usage", "Fused Mode", "Normalization", "Time Series Barycenters"):
    SoftDTW(gamma=1.0, fused=False, normalize=False)(x, y) -> (B,) losses, differentiable
    value_and_grad_host(x, y, gamma=1.0, fused=False) -> (loss, grad_x, grad_y) of a host batch
    soft_dtw_cost(C, gamma=1.0) -> (B,) losses of a given (B,N,M) cost, differentiable in C
    softdtw_barycenter(sequences, gamma=1.0, max_iter=100, lr=0.1, fused=True) -> (T, D)

PyTorch supplies device memory and streams only; every step of the method runs
in libsdtw.so's kernels.
"""
from __future__ import annotations

import math

import torch

from ._lib import (CHECKPOINT, EXTENDED, FUSED, OP_BARYCENTER, OP_COST, OP_FWD_BWD, OP_NORMALIZED, OP_NORMALIZED_UNEQUAL,
                   UNFUSED, SdtwError, sdtw_normalized_unequal, sdtw_normalized_backward,
                   sdtw_normalized_unequal_backward, sdtw_debug_set_options,
                   auto_precision, load, sdtw_backward, sdtw_backward_cost, sdtw_barycenter_step,
                   sdtw_backward_varlen, sdtw_barycenter_step_clipped, sdtw_debug_set_wait, sdtw_forward_varlen,
                   sdtw_distance, sdtw_forward, sdtw_forward_cost, sdtw_last_device_status, sdtw_normalized,
                   sdtw_workspace_bytes, workspace, host_workspace, sdtw_host_workspace_bytes,
                   sdtw_value_and_grad_host)

__all__ = [
    "SoftDTW", "soft_dtw_cost", "softdtw_barycenter", "SdtwError", "load", "workspace",
    "sdtw_workspace_bytes", "sdtw_distance", "sdtw_forward", "sdtw_backward", "sdtw_normalized",
    "sdtw_barycenter_step", "sdtw_barycenter_step_clipped", "sdtw_forward_cost", "sdtw_backward_cost",
    "sdtw_last_device_status", "cosine_lr", "sdtw_forward_varlen", "sdtw_backward_varlen",
    "sdtw_debug_set_wait", "UNFUSED", "FUSED", "EXTENDED", "OP_FWD_BWD", "OP_NORMALIZED", "OP_BARYCENTER",
    "OP_COST", "auto_precision", "value_and_grad_host", "host_workspace", "sdtw_host_workspace_bytes",
    "sdtw_value_and_grad_host", "sdtw_normalized_unequal", "OP_NORMALIZED_UNEQUAL", "CHECKPOINT",
    "sdtw_normalized_backward", "sdtw_normalized_unequal_backward", "sdtw_debug_set_options",
]


def _prep(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dim() != 3:
        raise ValueError(f"{name} must be (B, L, D)")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.detach().to(torch.float32).contiguous()


class _SoftDTWFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, y, gamma, mode):
        xc, yc = _prep(x, "x"), _prep(y, "y")
        if xc.shape[0] != yc.shape[0] or xc.shape[2] != yc.shape[2]:
            raise ValueError("x and y must share batch size and feature dimension")
        B, N, D = xc.shape
        M = yc.shape[1]
        ws = workspace(OP_FWD_BWD, B, N, M, D, mode, xc.device)
        loss = torch.empty(B, dtype=torch.float32, device=xc.device)
        sdtw_forward(xc, yc, gamma, mode, loss, ws)
        ctx.save_for_backward(xc, yc, ws)
        ctx.gamma, ctx.mode = gamma, mode
        ctx.dtypes = (x.dtype, y.dtype)
        return loss

    @staticmethod
    def backward(ctx, grad):
        xc, yc, ws = ctx.saved_tensors
        gx = torch.empty_like(xc) if ctx.needs_input_grad[0] else None
        gy = torch.empty_like(yc) if ctx.needs_input_grad[1] else None
        g = grad.detach().to(torch.float32).contiguous()
        sdtw_backward(xc, yc, ctx.gamma, ctx.mode, g, gx, gy, ws)
        return (None if gx is None else gx.to(ctx.dtypes[0]),
                None if gy is None else gy.to(ctx.dtypes[1]), None, None)


class _SoftDTWVarlenFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, y, x_lengths, y_lengths, gamma, mode):
        xc, yc = _prep(x, "x"), _prep(y, "y")
        if xc.shape[0] != yc.shape[0] or xc.shape[2] != yc.shape[2]:
            raise ValueError("x and y must share batch size and feature dimension")
        lx = None if x_lengths is None else x_lengths.to(device=xc.device, dtype=torch.int32).contiguous()
        ly = None if y_lengths is None else y_lengths.to(device=xc.device, dtype=torch.int32).contiguous()
        B, N, D = xc.shape
        M = yc.shape[1]
        ws = workspace(OP_FWD_BWD, B, N, M, D, mode, xc.device)
        loss = torch.empty(B, dtype=torch.float32, device=xc.device)
        sdtw_forward_varlen(xc, yc, lx, ly, gamma, mode, loss, ws)
        ctx.save_for_backward(xc, yc, ws)
        ctx.lens = (lx, ly)
        ctx.gamma, ctx.mode = gamma, mode
        ctx.dtypes = (x.dtype, y.dtype)
        return loss

    @staticmethod
    def backward(ctx, grad):
        xc, yc, ws = ctx.saved_tensors
        lx, ly = ctx.lens
        gx = torch.empty_like(xc) if ctx.needs_input_grad[0] else None
        gy = torch.empty_like(yc) if ctx.needs_input_grad[1] else None
        sdtw_backward_varlen(xc, yc, lx, ly, ctx.gamma, ctx.mode, grad.detach().to(torch.float32).contiguous(), gx,
                             gy, ws)
        return (None if gx is None else gx.to(ctx.dtypes[0]),
                None if gy is None else gy.to(ctx.dtypes[1]), None, None, None, None)


def _normalized_ws(xc, yc, mode):
    """Workspace of the normalized entry for these shapes: one batch of 3B
    (sdtw_normalized) at equal lengths, three batches of their own shapes
    (sdtw_normalized_unequal) otherwise."""
    B, N, D = xc.shape
    M = yc.shape[1]
    op = OP_NORMALIZED if N == M else OP_NORMALIZED_UNEQUAL
    return workspace(op, B, N, M, D, mode, xc.device)


class _NormalizedFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, y, gamma, mode):
        xc, yc = _prep(x, "x"), _prep(y, "y")
        if xc.shape[0] != yc.shape[0] or xc.shape[2] != yc.shape[2]:
            raise ValueError("normalized Soft-DTW needs x (B,N,D) and y (B,M,D)")
        loss = torch.empty(xc.shape[0], dtype=torch.float32, device=xc.device)
        ws = _normalized_ws(xc, yc, mode)
        if xc.shape[1] == yc.shape[1]:
            sdtw_normalized(xc, yc, gamma, mode, loss, None, None, None, ws)
        else:
            sdtw_normalized_unequal(xc, yc, gamma, mode, loss, None, None, None, ws)
        # the workspace holds the forward state of the three problems: the backward
        # runs from it without repeating the forward
        ctx.save_for_backward(xc, yc, ws)
        ctx.gamma, ctx.mode = gamma, mode
        ctx.dtypes = (x.dtype, y.dtype)
        return loss

    @staticmethod
    def backward(ctx, grad):
        xc, yc, ws = ctx.saved_tensors
        gx = torch.empty_like(xc) if ctx.needs_input_grad[0] else None
        gy = torch.empty_like(yc) if ctx.needs_input_grad[1] else None
        g = grad.detach().to(torch.float32).contiguous()
        if xc.shape[1] == yc.shape[1]:
            sdtw_normalized_backward(xc, yc, ctx.gamma, ctx.mode, g, gx, gy, ws)
        else:
            sdtw_normalized_unequal_backward(xc, yc, ctx.gamma, ctx.mode, g, gx, gy, ws)
        return (None if gx is None else gx.to(ctx.dtypes[0]),
                None if gy is None else gy.to(ctx.dtypes[1]), None, None)


class _CostFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, C, gamma, mode):
        Cc = C.detach().to(torch.float32).contiguous()
        if Cc.dim() != 3 or not Cc.is_cuda:
            raise ValueError("C must be a (B, N, M) CUDA tensor")
        B, N, M = Cc.shape
        ws = workspace(OP_COST, B, N, M, 1, mode, Cc.device)
        loss = torch.empty(B, dtype=torch.float32, device=Cc.device)
        sdtw_forward_cost(Cc, gamma, mode, loss, ws)
        ctx.save_for_backward(Cc, ws)
        ctx.gamma, ctx.mode, ctx.dtype = gamma, mode, C.dtype
        return loss

    @staticmethod
    def backward(ctx, grad):
        Cc, ws = ctx.saved_tensors
        gC = torch.empty_like(Cc)
        sdtw_backward_cost(Cc, ctx.gamma, ctx.mode, grad.detach().to(torch.float32).contiguous(), gC, ws)
        return gC.to(ctx.dtype), None, None


def soft_dtw_cost(C: torch.Tensor, gamma: float = 1.0, extended: bool | None = None) -> torch.Tensor:
    """Soft-DTW losses (B,) of a caller-supplied cost tensor C (B,N,M), for any
    discrepancy; differentiable in C (dL/dC = grad_loss * alignment matrix).
    extended=None picks the double-float DP state for small gamma or long
    sequences; True/False forces it."""
    if not (gamma > 0):
        raise ValueError("gamma must be > 0")
    if extended is None:
        mode = auto_precision(gamma, C.shape[1], C.shape[2])
    else:
        mode = EXTENDED if extended else 0
    return _CostFn.apply(C, float(gamma), mode)


class SoftDTW:
    """Per-pair Soft-DTW losses (B,), differentiable w.r.t. x and y.

    fused=False stores the (B,N,M) cost tensor; fused=True recomputes it inside
    the DP kernels. normalize=True gives s(x,y) - (s(x,x) + s(y,y))/2; x and y may
    differ in length. extended=None picks the double-float forward state unless
    the fp32 state is accurate enough for a batch-mean loss over these B pairs
    (auto_precision: small gamma, long sequences, D > 64, or D > 4 with B < 32
    select it); pass extended=True when the losses are summed rather than
    averaged. True/False forces it.
    checkpoint=True (fused, fp32, D <= 64, not normalized) keeps no per-cell forward
    state: the backward recomputes it band by band (128 rows) from the boundary rows
    the forward kept; the workspace holds one band, and the backward's time grows
    with the number of bands.
    """

    def __init__(self, gamma: float = 1.0, dist: str = "sqeuclidean", fused: bool = False,
                 normalize: bool = False, extended: bool | None = None, checkpoint: bool = False):
        if dist != "sqeuclidean":
            raise ValueError("only dist='sqeuclidean' is supported")
        if not (gamma > 0):
            raise ValueError("gamma must be > 0")
        if checkpoint and (not fused or normalize or extended):
            raise ValueError("checkpoint=True needs fused=True, normalize=False and the fp32 state")
        self.gamma = float(gamma)
        self.fused = bool(fused)
        self.normalize = normalize
        self.extended = extended
        self.checkpoint = bool(checkpoint)

    def __call__(self, x: torch.Tensor, y: torch.Tensor, x_lengths: torch.Tensor | None = None,
                 y_lengths: torch.Tensor | None = None) -> torch.Tensor:
        """x_lengths / y_lengths (B,) integer tensors make (x, y) a padded batch: pair b
        aligns x[b, :x_lengths[b]] with y[b, :y_lengths[b]]; padded rows get zero
        gradient and must be finite."""
        mode = FUSED if self.fused else UNFUSED
        if self.checkpoint:
            mode |= CHECKPOINT
        elif self.extended is None:
            mode |= auto_precision(self.gamma, x.shape[1], y.shape[1], x.shape[2], x.shape[0])
        elif self.extended:
            mode |= EXTENDED
        if x_lengths is not None or y_lengths is not None:
            if self.normalize:
                raise ValueError("normalize=True takes whole sequences, not a padded batch (x and y may differ in length)")
            return _SoftDTWVarlenFn.apply(x, y, x_lengths, y_lengths, self.gamma, mode)
        fn = _NormalizedFn if self.normalize else _SoftDTWFn
        return fn.apply(x, y, self.gamma, mode)


def value_and_grad_host(x: torch.Tensor, y: torch.Tensor, gamma: float = 1.0, fused: bool = False,
                        grad_loss: torch.Tensor | None = None, chunks: int = 2, extended: bool | None = None,
                        device=None):
    """Losses (B,) and input gradients of a batch held in host memory, in one call
    that overlaps the host<->device copies of one chunk of the batch with the
    kernels of the others. x (B,N,D), y (B,M,D) are float32 CPU tensors (pinned
    for overlap); grad_loss (B,) defaults to ones. Returns pinned CPU tensors
    (loss, grad_x, grad_y), complete when this function returns."""
    if not (gamma > 0):
        raise ValueError("gamma must be > 0")
    if x.dim() != 3 or y.dim() != 3 or x.shape[0] != y.shape[0] or x.shape[2] != y.shape[2]:
        raise ValueError("x must be (B,N,D) and y (B,M,D)")
    B, N, D = x.shape
    M = y.shape[1]
    mode = FUSED if fused else UNFUSED
    gl = torch.ones(B) if grad_loss is None else grad_loss.detach().to(torch.float32).contiguous()
    if extended is None:
        # the upstream weights are known here: the batch rule of auto_precision takes
        # the batch size whose mean would give the largest of them
        wmax = float(gl.abs().max()) if B > 0 else 1.0
        mode |= auto_precision(gamma, N, M, D, int(math.ceil(1.0 / wmax - 1e-6)) if wmax > 0 else B)
    elif extended:
        mode |= EXTENDED
    pin = torch.cuda.is_available()
    xh = x.detach().to(torch.float32).contiguous()
    yh = y.detach().to(torch.float32).contiguous()
    loss = torch.empty(B, pin_memory=pin)
    gx = torch.empty((B, N, D), pin_memory=pin)
    gy = torch.empty((B, M, D), pin_memory=pin)
    ws = host_workspace(B, N, M, D, mode, chunks, device=device)
    stream = torch.cuda.current_stream(ws.device)
    sdtw_value_and_grad_host(xh, yh, gl, gamma, mode, loss, gx, gy, chunks, ws, stream)
    code = sdtw_last_device_status(ws, stream)
    if code != 0:
        raise SdtwError(code, "value_and_grad_host")
    return loss, gx, gy


def cosine_lr(t: int, max_iter: int, lr: float, lr_min: float = 0.0) -> float:
    """Learning rate of step t (1-based) under cosine annealing from lr at t = 1
    to lr_min after max_iter steps, without restarts."""
    return lr_min + 0.5 * (lr - lr_min) * (1.0 + math.cos(math.pi * (t - 1) / max_iter))


def softdtw_barycenter(sequences: torch.Tensor, gamma: float = 1.0, max_iter: int = 100, lr: float = 0.1,
                       fused: bool = True, init: torch.Tensor | None = None, beta1: float = 0.9,
                       beta2: float = 0.999, eps: float = 1e-8, return_losses: bool = False,
                       lr_schedule: str | None = None, lr_min: float = 0.0, max_grad_norm: float | None = None,
                       early_stopping: bool = False, tol: float = 1e-4, patience: int = 10, check_every: int = 10):
    """Soft-DTW barycenter of K sequences (K,T,D) by Adam, initialised to their
    mean (or `init`), one sdtw_barycenter_step per iteration (README, "Time Series
    Barycenters"). Optional, as the README lists them (their parameters are not
    given there): lr_schedule="cosine" anneals the rate to lr_min over max_iter
    steps; max_grad_norm clips the gradient by its global L2 norm; early_stopping
    stops once the loss has not improved by more than tol * |best| for `patience`
    steps (losses are read back every `check_every` steps). Returns z, or
    (z, losses of the steps run) with return_losses."""
    X = _prep(sequences, "sequences")
    K, T2, D = X.shape
    z = (X.mean(dim=0) if init is None else init.detach().to(torch.float32)).contiguous().clone()
    T = z.shape[0]
    m = torch.zeros_like(z)
    v = torch.zeros_like(z)
    if lr_schedule not in (None, "cosine"):
        raise ValueError("lr_schedule must be None or 'cosine'")
    mode = (FUSED if fused else UNFUSED) | auto_precision(gamma, T, T2, D, K)   # the loss is the mean over K
    ws = workspace(OP_BARYCENTER, K, T, T2, D, mode, X.device)
    losses = torch.empty(max_iter, dtype=torch.float32, device=X.device)
    clip = float(max_grad_norm) if max_grad_norm else 0.0
    best, stale, ran = math.inf, 0, 0
    for t in range(1, max_iter + 1):
        lr_t = cosine_lr(t, max_iter, lr, lr_min) if lr_schedule == "cosine" else lr
        if clip > 0.0:
            sdtw_barycenter_step_clipped(z, m, v, t, X, gamma, lr_t, beta1, beta2, eps, clip, mode,
                                         losses[t - 1:t], ws)
        else:
            sdtw_barycenter_step(z, m, v, t, X, gamma, lr_t, beta1, beta2, eps, mode, losses[t - 1:t], ws)
        ran = t
        if early_stopping and (t % check_every == 0 or t == max_iter):
            for lv in losses[t - (t - 1) % check_every - 1:t].tolist():
                if lv < best - tol * abs(best) or best == math.inf:
                    best, stale = min(best, lv), 0
                else:
                    stale += 1
            if stale >= patience:
                break
    losses = losses[:ran]
    return (z, losses) if return_losses else z
