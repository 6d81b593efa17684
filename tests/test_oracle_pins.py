"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle.

Each test checks the oracle against something other than itself -- closed
forms, brute-force enumeration of every warping path, hard DTW, finite
differences, invariants -- chosen so that a dropped term, a wrong sign, a
wrong index or a transposed operand in the oracle fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from differentiable_series_alignment_gb300 import synth

RNG = np.random.default_rng(1234)


def _pair(N, M, D, scale=1.0, seed=0):
    g = np.random.default_rng(seed)
    return (scale * g.standard_normal((N, D))), (scale * g.standard_normal((M, D)))


def _cost(x, y):
    # Written independently of the oracle: explicit loops.
    N, M = len(x), len(y)
    C = np.zeros((N, M))
    for i in range(N):
        for j in range(M):
            C[i, j] = float(np.sum((np.asarray(x[i]) - np.asarray(y[j])) ** 2))
    return C


def _paths(N, M):
    """All monotone warping paths from (0,0) to (N-1,M-1) with unit steps
    right, down and diagonal."""
    out = []

    def rec(i, j, acc):
        if i == N - 1 and j == M - 1:
            out.append(list(acc))
            return
        for di, dj in ((1, 0), (0, 1), (1, 1)):
            a, b = i + di, j + dj
            if a < N and b < M:
                acc.append((a, b))
                rec(a, b, acc)
                acc.pop()

    rec(0, 0, [(0, 0)])
    return out


def _delannoy(n, m):
    return sum(math.comb(m, k) * math.comb(n, k) * 2 ** k for k in range(min(n, m) + 1))


def _brute(C, gamma):
    N, M = C.shape
    P = _paths(N, M)
    costs = np.array([sum(C[a, b] for a, b in p) for p in P])
    z = -costs / gamma
    zmax = z.max()
    w = np.exp(z - zmax)
    Z = w.sum()
    R = -gamma * (zmax + math.log(Z))
    E = np.zeros((N, M))
    for p, wp in zip(P, w / Z):
        for a, b in p:
            E[a, b] += wp
    return R, E, len(P)


def _hard_dtw(C):
    N, M = C.shape
    R = np.full((N + 1, M + 1), np.inf)
    R[0, 0] = 0.0
    for i in range(1, N + 1):
        for j in range(1, M + 1):
            R[i, j] = C[i - 1, j - 1] + min(R[i - 1, j - 1], R[i - 1, j], R[i, j - 1])
    return R[N, M]


# --------------------------------------------------------------------------- closed forms

def test_single_cell_is_the_distance():
    x, y = _pair(1, 1, 5, seed=1)
    out = oracle.single(x, y, 0.7, want_E=True)
    assert out["loss"] == pytest.approx(float(np.sum((x - y) ** 2)), rel=1e-14)
    np.testing.assert_allclose(out["E"], [[1.0]], rtol=0, atol=1e-14)


@pytest.mark.parametrize("N,M", [(1, 9), (7, 1)])
def test_single_row_or_column_is_a_plain_sum(N, M):
    x, y = _pair(N, M, 3, seed=2)
    out = oracle.single(x, y, 0.3, want_E=True)
    C = _cost(x, y)
    assert out["loss"] == pytest.approx(C.sum(), rel=1e-13)
    np.testing.assert_allclose(out["E"], np.ones((N, M)), rtol=0, atol=1e-12)


def test_two_by_two_closed_form():
    x, y = _pair(2, 2, 4, seed=3)
    C = _cost(x, y)
    g = 1.3
    expect = C[0, 0] + C[1, 1] - g * math.log(1 + math.exp(-C[0, 1] / g) + math.exp(-C[1, 0] / g))
    assert oracle.single(x, y, g)["loss"] == pytest.approx(expect, rel=1e-13)


# --------------------------------------------------------------------------- brute force

def test_path_enumerator_counts_are_delannoy_numbers():
    for n in range(1, 6):
        assert len(_paths(n, n)) == _delannoy(n - 1, n - 1)
    assert [_delannoy(n, n) for n in range(7)] == [1, 3, 13, 63, 321, 1683, 8989]


@pytest.mark.parametrize("N,M,gamma,seed", [(3, 3, 1.0, 4), (4, 6, 0.5, 5), (6, 5, 2.0, 6),
                                            (6, 6, 0.1, 7), (2, 7, 1.0, 8)])
def test_brute_force_value_and_alignment(N, M, gamma, seed):
    x, y = _pair(N, M, 3, scale=0.6, seed=seed)
    C = _cost(x, y)
    Rb, Eb, npaths = _brute(C, gamma)
    assert npaths == _delannoy(N - 1, M - 1)
    out = oracle.single(x, y, gamma, want_E=True)
    assert out["loss"] == pytest.approx(Rb, rel=1e-12, abs=1e-12)
    np.testing.assert_allclose(out["E"], Eb, rtol=1e-10, atol=1e-13)


def test_brute_force_on_a_given_cost_matrix():
    # Cost matrix with distinct entries, so a transposed operand would show.
    C = np.arange(1, 21, dtype=np.float64).reshape(4, 5) / 7.0
    C[1, 3] = 0.05
    Rb, Eb, _ = _brute(C, 0.8)
    R = oracle.forward_from_cost(C, 0.8)
    assert R[4, 5] == pytest.approx(Rb, rel=1e-13)
    np.testing.assert_allclose(oracle.backward_from_cost(C, R, 0.8), Eb, rtol=1e-11, atol=1e-14)


# --------------------------------------------------------------------------- gamma -> 0

@pytest.mark.parametrize("gamma", [1.0, 0.1, 0.01, 1e-3])
def test_sandwich_between_hard_dtw_bounds(gamma):
    N, M = 9, 11
    x, y = _pair(N, M, 2, seed=9)
    C = _cost(x, y)
    dtw = _hard_dtw(C)
    R = oracle.single(x, y, gamma)["loss"]
    assert R <= dtw + 1e-12
    assert R >= dtw - gamma * math.log(_delannoy(N - 1, M - 1)) - 1e-12


def test_small_gamma_alignment_is_the_optimal_path():
    N, M = 8, 8
    x, y = _pair(N, M, 2, seed=10)
    C = _cost(x, y)
    # optimal hard path by explicit back-tracking
    R = np.full((N + 1, M + 1), np.inf)
    R[0, 0] = 0
    for i in range(1, N + 1):
        for j in range(1, M + 1):
            R[i, j] = C[i - 1, j - 1] + min(R[i - 1, j - 1], R[i - 1, j], R[i, j - 1])
    A = np.zeros((N, M))
    i, j = N, M
    while (i, j) != (0, 0):
        A[i - 1, j - 1] = 1
        cands = [(R[i - 1, j - 1], i - 1, j - 1), (R[i - 1, j], i - 1, j), (R[i, j - 1], i, j - 1)]
        _, i, j = min(cands)
    out = oracle.single(x, y, 1e-3, want_E=True)
    np.testing.assert_allclose(out["E"], A, atol=1e-6)


# --------------------------------------------------------------------------- derivatives

def test_alignment_is_the_derivative_wrt_cost():
    g = np.random.default_rng(11)
    C = g.uniform(0.1, 3.0, size=(5, 6))
    gamma = 0.7
    E = oracle.backward_from_cost(C, oracle.forward_from_cost(C, gamma), gamma)
    h = 1e-6
    fd = np.zeros_like(C)
    for idx in np.ndindex(C.shape):
        Cp, Cm = C.copy(), C.copy()
        Cp[idx] += h
        Cm[idx] -= h
        fd[idx] = (oracle.forward_from_cost(Cp, gamma)[-1, -1]
                   - oracle.forward_from_cost(Cm, gamma)[-1, -1]) / (2 * h)
    np.testing.assert_allclose(E, fd, rtol=1e-7, atol=1e-9)


@pytest.mark.parametrize("N,M,D,gamma", [(5, 6, 3, 1.0), (7, 4, 2, 0.2)])
def test_input_gradients_match_central_differences(N, M, D, gamma):
    x, y = _pair(N, M, D, seed=12)
    gl = 0.37
    out = oracle.single(x, y, gamma, g=gl)
    h = 1e-6

    def f(xx, yy):
        return gl * oracle.single(xx, yy, gamma)["loss"]

    fdx = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fdx[idx] = (f(xp, y) - f(xm, y)) / (2 * h)
    fdy = np.zeros_like(y)
    for idx in np.ndindex(y.shape):
        yp, ym = y.copy(), y.copy()
        yp[idx] += h
        ym[idx] -= h
        fdy[idx] = (f(x, yp) - f(x, ym)) / (2 * h)
    np.testing.assert_allclose(out["gx"], fdx, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(out["gy"], fdy, rtol=1e-6, atol=1e-8)


# --------------------------------------------------------------------------- invariants

def test_symmetry_swaps_gradients():
    x, y = _pair(6, 9, 3, seed=13)
    a = oracle.single(x, y, 0.9)
    b = oracle.single(y, x, 0.9)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-13)
    np.testing.assert_allclose(a["gx"], b["gy"], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(a["gy"], b["gx"], rtol=1e-11, atol=1e-13)


def test_time_reversal_invariance():
    x, y = _pair(8, 6, 2, seed=14)
    a = oracle.single(x, y, 0.5)
    b = oracle.single(x[::-1], y[::-1], 0.5)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-12)
    np.testing.assert_allclose(a["gx"], b["gx"][::-1], rtol=1e-10, atol=1e-12)


def test_homogeneity():
    x, y = _pair(7, 7, 3, seed=15)
    alpha, gamma = 1.7, 0.6
    a = oracle.single(alpha * x, alpha * y, gamma)["loss"]
    b = oracle.single(x, y, gamma / alpha ** 2)["loss"]
    assert a == pytest.approx(alpha ** 2 * b, rel=1e-12)


def test_alignment_bounds_and_marginals():
    x, y = _pair(10, 13, 3, seed=16)
    E = oracle.single(x, y, 0.8, want_E=True)["E"]
    assert E.min() > 0 and E.max() <= 1 + 1e-12
    assert E[0, 0] == pytest.approx(1.0, abs=1e-12)
    assert E[-1, -1] == pytest.approx(1.0, abs=1e-12)
    # every monotone path visits each row and each column at least once
    assert np.all(E.sum(axis=1) >= 1 - 1e-12)
    assert np.all(E.sum(axis=0) >= 1 - 1e-12)


def test_entropy_identity():
    """Soft-DTW = expected cost minus gamma times the entropy of the path
    distribution, the entropy taken as a sum over cells of the visit
    probability times the entropy of that cell's predecessor choice."""
    x, y = _pair(7, 9, 2, seed=17)
    gamma = 0.8
    out = oracle.single(x, y, gamma, want_R=True, want_E=True)
    R, E = out["R"], out["E"]
    C = _cost(x, y)
    N, M = C.shape
    H = 0.0
    for i in range(1, N + 1):
        for j in range(1, M + 1):
            preds = [(i - 1, j - 1), (i - 1, j), (i, j - 1)]
            ps = [math.exp((R[i, j] - C[i - 1, j - 1] - R[a, b]) / gamma)
                  for a, b in preds if np.isfinite(R[a, b])]
            assert sum(ps) == pytest.approx(1.0, abs=1e-12)
            H += E[i - 1, j - 1] * -sum(p * math.log(p) for p in ps if p > 0)
    assert R[N, M] == pytest.approx(float(np.sum(E * C)) - gamma * H, rel=1e-11)


def test_value_can_be_negative():
    x = np.zeros((6, 1))
    y = np.zeros((6, 1))
    assert oracle.single(x, y, 1.0)["loss"] < 0


# --------------------------------------------------------------------------- normalized

def test_normalized_is_zero_with_zero_gradient_at_equal_inputs():
    g = np.random.default_rng(18)
    x = g.standard_normal((3, 12, 4))
    loss, gx, gy = oracle.normalized(x, x, 0.7, grad_loss=np.ones(3))
    np.testing.assert_allclose(loss, 0.0, atol=1e-12)
    np.testing.assert_allclose(gx, 0.0, atol=1e-10)
    np.testing.assert_allclose(gy, 0.0, atol=1e-10)


def test_normalized_gradient_matches_central_differences():
    g = np.random.default_rng(19)
    x = g.standard_normal((1, 5, 2))
    y = g.standard_normal((1, 5, 2))
    gamma = 0.9
    _, gx, gy = oracle.normalized(x, y, gamma, grad_loss=[1.0])
    h = 1e-6

    def f(a, b):
        return oracle.normalized(a, b, gamma)[0][0]

    for arr, grad, first in ((x, gx, True), (y, gy, False)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            fd[idx] = ((f(p, y) - f(m, y)) if first else (f(x, p) - f(x, m))) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)


def test_normalized_matches_three_separate_values():
    g = np.random.default_rng(20)
    x = g.standard_normal((2, 6, 3))
    y = g.standard_normal((2, 6, 3))
    loss, _, _ = oracle.normalized(x, y, 0.5)
    for b in range(2):
        s = lambda a, c: _brute(_cost(a, c), 0.5)[0]
        expect = s(x[b], y[b]) - 0.5 * (s(x[b], x[b]) + s(y[b], y[b]))
        assert loss[b] == pytest.approx(expect, rel=1e-10, abs=1e-10)


def test_unequal_normalized_reduces_to_the_equal_length_oracle():
    # at N == M the composed definition must agree with the C oracle's own normalized
    g = np.random.default_rng(40)
    x = g.standard_normal((3, 9, 2))
    y = g.standard_normal((3, 9, 2))
    w = np.array([0.5, -1.0, 2.0])
    l1, gx1, gy1 = oracle.normalized(x, y, 0.8, grad_loss=w)
    l2, gx2, gy2 = oracle.normalized_unequal(x, y, 0.8, grad_loss=w)
    np.testing.assert_allclose(l2, l1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gx2, gx1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gy2, gy1, rtol=1e-10, atol=1e-12)


def test_unequal_normalized_values_by_brute_force():
    g = np.random.default_rng(41)
    x = g.standard_normal((2, 6, 3))
    y = g.standard_normal((2, 4, 3))
    loss, _, _ = oracle.normalized_unequal(x, y, 0.6)
    for b in range(2):
        s = lambda a, c: _brute(_cost(a, c), 0.6)[0]
        expect = s(x[b], y[b]) - 0.5 * (s(x[b], x[b]) + s(y[b], y[b]))
        assert loss[b] == pytest.approx(expect, rel=1e-10, abs=1e-10)


def test_unequal_normalized_is_symmetric_with_gradients_swapped():
    g = np.random.default_rng(42)
    x = g.standard_normal((2, 7, 2))
    y = g.standard_normal((2, 4, 2))
    w = np.array([1.0, -0.5])
    l1, gx1, gy1 = oracle.normalized_unequal(x, y, 0.9, grad_loss=w)
    l2, gx2, gy2 = oracle.normalized_unequal(y, x, 0.9, grad_loss=w)
    np.testing.assert_allclose(l2, l1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gx2, gy1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gy2, gx1, rtol=1e-10, atol=1e-12)


def test_unequal_normalized_gradient_matches_central_differences():
    g = np.random.default_rng(43)
    x = g.standard_normal((1, 5, 2))
    y = g.standard_normal((1, 3, 2))
    gamma = 0.7
    _, gx, gy = oracle.normalized_unequal(x, y, gamma, grad_loss=[1.0])
    h = 1e-6

    def f(a, b):
        return oracle.normalized_unequal(a, b, gamma)[0][0]

    for arr, grad, first in ((x, gx, True), (y, gy, False)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            fd[idx] = ((f(p, y) - f(m, y)) if first else (f(x, p) - f(x, m))) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)


# --------------------------------------------------------------------------- barycenter step

def test_adam_first_step_moves_each_coordinate_by_lr_against_the_gradient():
    g = np.random.default_rng(21)
    X = g.standard_normal((4, 7, 2))
    z = X.mean(axis=0)
    z1, m, v, loss, grad = oracle.barycenter_step(z, np.zeros_like(z), np.zeros_like(z), 1, X,
                                                  gamma=1.0, lr=0.1)
    big = np.abs(grad) > 1e-3
    np.testing.assert_allclose((z1 - z)[big], -0.1 * np.sign(grad[big]), rtol=1e-4)


def test_barycenter_gradient_is_the_derivative_of_the_mean_loss():
    g = np.random.default_rng(22)
    X = g.standard_normal((3, 6, 2))
    z = g.standard_normal((5, 2))
    _, _, _, loss, grad = oracle.barycenter_step(z, np.zeros_like(z), np.zeros_like(z), 1, X, 0.8)

    def f(zz):
        return float(np.mean([_brute(_cost(zz, X[k]), 0.8)[0] for k in range(3)]))

    assert loss == pytest.approx(f(z), rel=1e-10)
    h = 1e-6
    fd = np.zeros_like(z)
    for idx in np.ndindex(z.shape):
        p, m = z.copy(), z.copy()
        p[idx] += h
        m[idx] -= h
        fd[idx] = (f(p) - f(m)) / (2 * h)
    np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)


def test_barycenter_constant_gradient_steps_are_lr_sized():
    # With a gradient of constant sign, every bias-corrected Adam step has size ~lr.
    g = np.random.default_rng(23)
    X = g.standard_normal((2, 6, 1)) + 5.0   # sequences far above z, gradient sign stays fixed
    z = np.zeros((6, 1))
    m = np.zeros_like(z)
    v = np.zeros_like(z)
    for t in range(1, 4):
        z_new, m, v, _, grad = oracle.barycenter_step(z, m, v, t, X, 1.0, lr=0.05)
        assert np.all(grad < 0)
        np.testing.assert_allclose(z_new - z, 0.05, rtol=2e-2)
        z = z_new


# --------------------------------------------------------------------------- batch wrapper

def test_batch_equals_single_per_problem():
    g = np.random.default_rng(24)
    x = g.standard_normal((3, 5, 2)).astype(np.float32)
    y = g.standard_normal((3, 4, 2)).astype(np.float32)
    gl = np.array([0.5, -1.0, 2.0])
    loss, gx, gy = oracle.batch(x, y, 0.6, grad_loss=gl)
    for b in range(3):
        s = oracle.single(x[b], y[b], 0.6, g=gl[b])
        assert loss[b] == s["loss"]
        np.testing.assert_array_equal(gx[b], s["gx"])
        np.testing.assert_array_equal(gy[b], s["gy"])


def test_barycenter_gradient_clipping_pins():
    """Clipping by the global L2 norm: a bound at or above ||g|| changes nothing,
    and below it the first step's moments carry exactly the clipped norm
    (m = (1-b1) g c/||g||, v = (1-b2) (g c/||g||)^2), while the first Adam step
    itself is scale-free."""
    X = synth.block_waves(4, 24, 2, 4)
    z = X.astype(np.float64).mean(axis=0)
    zero = np.zeros_like(z)
    z1, m1, v1, l1, g = oracle.barycenter_step(z, zero, zero, 1, X, 1.0)
    nrm = float(np.linalg.norm(g))
    assert nrm > 0
    za, ma, va, la, ga = oracle.barycenter_step(z, zero, zero, 1, X, 1.0, max_grad_norm=nrm * 1.0001)
    assert np.array_equal(za, z1) and np.array_equal(ma, m1) and np.array_equal(va, v1) and la == l1
    c = 0.25 * nrm
    zc, mc, vc, lc, gc = oracle.barycenter_step(z, zero, zero, 1, X, 1.0, max_grad_norm=c)
    assert np.array_equal(gc, g)                                  # the raw gradient is returned
    assert np.linalg.norm(mc) == pytest.approx(0.1 * c, rel=1e-12)
    assert vc.sum() == pytest.approx(0.001 * c * c, rel=1e-12)
    np.testing.assert_allclose(zc, z1, rtol=0, atol=1e-6)         # step 1 moves lr*sign(g) either way
