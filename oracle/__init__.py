"""fp64 CPU oracle for batched Soft-DTW -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this package. The CUDA library never calls it and shares no
code with it. The arithmetic lives in ``sdtw_oracle.c`` (plain C, double
precision); this module compiles it with gcc on first use and wraps it with
ctypes. Inputs are converted to float64 exactly (float32 -> float64 is exact),
so the oracle sees the very values the CUDA path sees. ``normalized_unequal``
composes three ``batch`` calls in Python (its definition, term by term).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdtw_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc -O2, OpenMP) if it is stale."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_single.argtypes = [_dp, _dp, i, i, i, d, d, _dp, _dp, _dp, _dp, _dp]
            lib.oracle_single.restype = i
            lib.oracle_batch.argtypes = [_dp, _dp, i, i, i, i, d, _dp, _dp, _dp, _dp, i]
            lib.oracle_batch.restype = i
            lib.oracle_normalized.argtypes = [_dp, _dp, i, i, i, d, _dp, _dp, _dp, _dp, i]
            lib.oracle_normalized.restype = i
            lib.oracle_barycenter_step.argtypes = [_dp, _dp, _dp, i, _dp, i, i, i, i, d, d, d, d, d,
                                                   d, _dp, _dp, i]
            lib.oracle_barycenter_step.restype = i
            lib.oracle_forward.argtypes = [_dp, i, i, d, _dp]
            lib.oracle_forward.restype = d
            lib.oracle_backward.argtypes = [_dp, _dp, i, i, d, _dp]
            lib.oracle_backward.restype = None
            lib.oracle_threads_used.argtypes = [i]
            lib.oracle_threads_used.restype = i
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def threads_used(nthreads: int = 0) -> int:
    return _load().oracle_threads_used(int(nthreads))


def single(x, y, gamma, g=1.0, want_R=False, want_E=False):
    """One problem: x (N,D), y (M,D). Returns dict(loss, gx, gy[, R, E])."""
    x, y = _f64(x), _f64(y)
    N, D = x.shape
    M = y.shape[0]
    gx = np.empty((N, D))
    gy = np.empty((M, D))
    R = np.empty((N + 1, M + 1)) if want_R else None
    E = np.empty((N, M)) if want_E else None
    loss = ctypes.c_double()
    rc = _load().oracle_single(_ptr(x), _ptr(y), N, M, D, float(gamma), float(g),
                               ctypes.byref(loss), _ptr(gx), _ptr(gy), _ptr(R), _ptr(E))
    if rc != 0:
        raise ValueError("oracle_single: bad argument")
    out = dict(loss=loss.value, gx=gx, gy=gy)
    if want_R:
        out["R"] = R
    if want_E:
        out["E"] = E
    return out


def forward_from_cost(C, gamma):
    """R ((N+1),(M+1)) for a given cost matrix C (N,M)."""
    C = _f64(C)
    N, M = C.shape
    R = np.empty((N + 1, M + 1))
    _load().oracle_forward(_ptr(C), N, M, float(gamma), _ptr(R))
    return R


def backward_from_cost(C, R, gamma):
    """E (N,M) for a cost matrix C and its forward table R."""
    C, R = _f64(C), _f64(R)
    N, M = C.shape
    E = np.empty((N, M))
    _load().oracle_backward(_ptr(C), _ptr(R), N, M, float(gamma), _ptr(E))
    return E


def batch(x, y, gamma, grad_loss=None, nthreads=0):
    """B problems: x (B,N,D), y (B,M,D). Returns (loss (B,), gx, gy)."""
    x, y = _f64(x), _f64(y)
    B, N, D = x.shape
    M = y.shape[1]
    loss = np.empty(B)
    gl = None if grad_loss is None else _f64(np.broadcast_to(np.asarray(grad_loss, np.float64), (B,)))
    gx = np.empty_like(x) if gl is not None else None
    gy = np.empty_like(y) if gl is not None else None
    rc = _load().oracle_batch(_ptr(x), _ptr(y), B, N, M, D, float(gamma), _ptr(gl), _ptr(loss),
                              _ptr(gx), _ptr(gy), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_batch: bad argument or allocation failure")
    return loss, gx, gy


def normalized(x, y, gamma, grad_loss=None, nthreads=0):
    """Normalized Soft-DTW over B pairs of equal shape (B,N,D)."""
    x, y = _f64(x), _f64(y)
    if x.shape != y.shape:
        raise ValueError("normalized Soft-DTW needs x.shape == y.shape")
    B, N, D = x.shape
    loss = np.empty(B)
    gl = None if grad_loss is None else _f64(np.broadcast_to(np.asarray(grad_loss, np.float64), (B,)))
    gx = np.empty_like(x) if gl is not None else None
    gy = np.empty_like(y) if gl is not None else None
    rc = _load().oracle_normalized(_ptr(x), _ptr(y), B, N, D, float(gamma), _ptr(gl), _ptr(loss),
                                   _ptr(gx), _ptr(gy), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_normalized: bad argument or allocation failure")
    return loss, gx, gy


def normalized_unequal(x, y, gamma, grad_loss=None, nthreads=0):
    """Normalized Soft-DTW of pairs whose sequences differ in length, x (B,N,D) and
    y (B,M,D): the definition of the SoftDTW README's "Normalization" section,
    s(x,y) - (s(x,x) + s(y,y))/2, applied unchanged to N != M, with the three
    terms from `batch`:
        grad_x = g [gx(x,y) - (gx(x,x) + gy(x,x))/2]
        grad_y = g [gy(x,y) - (gx(y,y) + gy(y,y))/2]
    (x sits in both slots of s(x,x), so both of its gradients count)."""
    x, y = _f64(x), _f64(y)
    if x.ndim != 3 or y.ndim != 3 or x.shape[0] != y.shape[0] or x.shape[2] != y.shape[2]:
        raise ValueError("x must be (B,N,D) and y (B,M,D)")
    lxy, gxy_x, gxy_y = batch(x, y, gamma, grad_loss=grad_loss, nthreads=nthreads)
    lxx, gxx_x, gxx_y = batch(x, x, gamma, grad_loss=grad_loss, nthreads=nthreads)
    lyy, gyy_x, gyy_y = batch(y, y, gamma, grad_loss=grad_loss, nthreads=nthreads)
    loss = lxy - 0.5 * (lxx + lyy)
    if grad_loss is None:
        return loss, None, None
    return loss, gxy_x - 0.5 * (gxx_x + gxx_y), gxy_y - 0.5 * (gyy_x + gyy_y)


def barycenter_step(z, m, v, t, X, gamma, lr=0.1, beta1=0.9, beta2=0.999, eps=1e-8, nthreads=0,
                    max_grad_norm=0.0):
    """One Adam step; returns (z, m, v, loss_at_incoming_z, grad) as new arrays.
    max_grad_norm > 0 clips the gradient by its global L2 norm before Adam; the
    returned grad is the unclipped one."""
    z, m, v, X = _f64(z).copy(), _f64(m).copy(), _f64(v).copy(), _f64(X)
    T, D = z.shape
    K, T2, _ = X.shape
    loss = ctypes.c_double()
    grad = np.empty_like(z)
    rc = _load().oracle_barycenter_step(_ptr(z), _ptr(m), _ptr(v), int(t), _ptr(X), K, T, T2, D,
                                        float(gamma), float(lr), float(beta1), float(beta2),
                                        float(eps), float(max_grad_norm), ctypes.byref(loss), _ptr(grad),
                                        int(nthreads))
    if rc != 0:
        raise ValueError("oracle_barycenter_step: bad argument or allocation failure")
    return z, m, v, loss.value, grad
